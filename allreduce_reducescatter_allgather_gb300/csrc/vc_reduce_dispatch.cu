// From a run-time (element type, op, order) to the slice that holds its
// kernels.
//
// Integer results do not depend on the reduction order: the ops wrap modulo
// 2^64 (SUM, PROD) or pick one of the operands (MAX, MIN), all exactly
// associative and commutative, so every order gives the same bits.  The
// integer types therefore run every order on the ring's kernels, the
// fastest at every N, and have no tree or recursive-halving instances.
#include "vc_launch.cuh"

namespace vc {

#define VC_DECLARE_OP(ty, op)                                                                  \
    cudaError_t launch_reduce_##ty##_##op##_g0(const ReduceParams&, int, bool, cudaStream_t); \
    cudaError_t launch_reduce_##ty##_##op##_g1(const ReduceParams&, int, bool, cudaStream_t); \
    cudaError_t launch_reduce_##ty##_##op##_g2(const ReduceParams&, int, bool, cudaStream_t); \
    static cudaError_t launch_reduce_##ty##_##op(const ReduceParams& p, int order, bool rs,     \
                                                 cudaStream_t st) {                            \
        switch (order_group(order, p.n)) {                                                     \
        case kGroupRingRh: return launch_reduce_##ty##_##op##_g0(p, order, rs, st);            \
        case kGroupTree: return launch_reduce_##ty##_##op##_g1(p, order, rs, st);              \
        default: return launch_reduce_##ty##_##op##_g2(p, order, rs, st);                      \
        }                                                                                      \
    }
#define VC_DECLARE_INT_OP(ty, op)                                                              \
    cudaError_t launch_reduce_##ty##_##op##_g0(const ReduceParams&, int, bool, cudaStream_t); \
    static cudaError_t launch_reduce_##ty##_##op(const ReduceParams& p, int, bool rs,          \
                                                 cudaStream_t st) {                            \
        return launch_reduce_##ty##_##op##_g0(p, kOrderRing, rs, st);                          \
    }
#define VC_DECLARE(ty, D) \
    D(ty, sum)            \
    D(ty, prod)           \
    D(ty, max)            \
    D(ty, min)
VC_DECLARE(i32, VC_DECLARE_INT_OP)
VC_DECLARE(i64, VC_DECLARE_INT_OP)
VC_DECLARE(f32, VC_DECLARE_OP)
VC_DECLARE(bf16, VC_DECLARE_OP)
#undef VC_DECLARE
#undef VC_DECLARE_OP
#undef VC_DECLARE_INT_OP

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
