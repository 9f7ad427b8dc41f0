// ReduceScatter / AllReduce kernel instances for element type __nv_bfloat16.
#include "vc_launch.cuh"

namespace vc {
cudaError_t launch_reduce_bf16(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st) {
    return launch_reduce_t<__nv_bfloat16>(p, op, order, rs, st);
}
}  // namespace vc
