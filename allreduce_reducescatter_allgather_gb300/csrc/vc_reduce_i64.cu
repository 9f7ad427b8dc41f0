// ReduceScatter / AllReduce kernel instances for element type long long.
#include "vc_launch.cuh"

namespace vc {
cudaError_t launch_reduce_i64(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st) {
    return launch_reduce_t<long long>(p, op, order, rs, st);
}
}  // namespace vc
