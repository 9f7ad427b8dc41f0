// From a run-time (element type, op) to the slice that holds its kernels.
#include "vc_device.cuh"

namespace vc {

#define VC_DECLARE(ty)                                                                       \
    cudaError_t launch_reduce_##ty##_sum(const ReduceParams&, int, bool, cudaStream_t);  \
    cudaError_t launch_reduce_##ty##_prod(const ReduceParams&, int, bool, cudaStream_t); \
    cudaError_t launch_reduce_##ty##_max(const ReduceParams&, int, bool, cudaStream_t);  \
    cudaError_t launch_reduce_##ty##_min(const ReduceParams&, int, bool, cudaStream_t);
VC_DECLARE(i32)
VC_DECLARE(i64)
VC_DECLARE(f32)
VC_DECLARE(bf16)
#undef VC_DECLARE

// op: 0 sum, 1 prod, 2 max, 3 min, 4 avg (the sum kernels with p.avg set)
#define VC_DISPATCH(ty)                                                                         \
    cudaError_t launch_reduce_##ty(const ReduceParams& p, int op, int order, bool rs,          \
                                   cudaStream_t st) {                                          \
        switch (op) {                                                                          \
        case 0:                                                                                \
        case 4: return launch_reduce_##ty##_sum(p, order, rs, st);                             \
        case 1: return launch_reduce_##ty##_prod(p, order, rs, st);                            \
        case 2: return launch_reduce_##ty##_max(p, order, rs, st);                             \
        case 3: return launch_reduce_##ty##_min(p, order, rs, st);                             \
        default: return cudaErrorInvalidValue;                                                 \
        }                                                                                      \
    }
VC_DISPATCH(i32)
VC_DISPATCH(i64)
VC_DISPATCH(f32)
VC_DISPATCH(bf16)
#undef VC_DISPATCH

}  // namespace vc
