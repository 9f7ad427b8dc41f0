// One element type's slice of the fused bucket kernels.  The
// build compiles this file once per type, with
//   -DVC_T=<element type> -DVC_FN=<launcher name>.
#include "vc_bucket_kernel.cuh"

#if !defined(VC_T) || !defined(VC_FN)
#error "compile with -DVC_T=... -DVC_FN=..."
#endif

namespace vc {
cudaError_t VC_FN(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st) {
    return launch_bucket_op<VC_T>(p, op, rs, st);
}
}  // namespace vc
