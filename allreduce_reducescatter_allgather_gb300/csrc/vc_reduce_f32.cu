// ReduceScatter / AllReduce kernel instances for element type float.
#include "vc_launch.cuh"

namespace vc {
cudaError_t launch_reduce_f32(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st) {
    return launch_reduce_t<float>(p, op, order, rs, st);
}
}  // namespace vc
