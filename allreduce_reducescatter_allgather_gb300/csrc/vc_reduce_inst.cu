// One (element type, op, order group) slice of the ReduceScatter /
// AllReduce kernel instances.  The build compiles this file once per triple,
// with
//   -DVC_T=<element type> -DVC_OP=<op functor> -DVC_GROUP=<order group>
//   -DVC_FN=<launcher name>,
// so the slices compile in parallel.
#include "vc_launch.cuh"

#if !defined(VC_T) || !defined(VC_OP) || !defined(VC_GROUP) || !defined(VC_FN)
#error "compile with -DVC_T=... -DVC_OP=... -DVC_GROUP=... -DVC_FN=..."
#endif

namespace vc {
cudaError_t VC_FN(const ReduceParams& p, int order, bool rs, cudaStream_t st) {
    return launch_group<VC_T, VC_OP, VC_GROUP>(p, order, rs, st);
}
}  // namespace vc
