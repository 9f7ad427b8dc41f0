// ReduceScatter / AllReduce kernel instances for element type int32_t.
#include "vc_launch.cuh"

namespace vc {
cudaError_t launch_reduce_i32(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st) {
    return launch_reduce_t<int32_t>(p, op, order, rs, st);
}
}  // namespace vc
