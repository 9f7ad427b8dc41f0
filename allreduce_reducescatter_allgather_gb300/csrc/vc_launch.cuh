// Dispatch from a run-time (order, N) to a kernel instance.  Included by
// vc_reduce_inst.cu, which the build compiles once per (element type, op,
// order group), and by vc_reduce_dispatch.cu for order_group().
#pragma once

#include "vc_device.cuh"

namespace vc {

// Programmatic dependent launch (launch_pdl): the grid may be scheduled
// while the kernel before it on the stream drains (the kernels wait on
// griddepcontrol before their first global access, and signal their
// dependents as each block finishes), so back-to-back collectives do not pay
// the full launch gap.
template <class T, class Op, int ORDER, int NT, int U>
cudaError_t launch_one(const ReduceParams& p, bool rs, cudaStream_t st) {
    constexpr int V = Traits<T>::V;
    const long long nvec = (p.limit + V - 1) / V;
    const int blocks = grid_blocks((nvec + U - 1) / U);
    if (blocks < 1) return cudaErrorInvalidConfiguration;
    if (rs) return launch_pdl(vc_rs_kernel<T, Op, ORDER, NT, U>, dim3(blocks), dim3(kThreads), st, p);
    return launch_pdl(vc_ar_kernel<T, Op, ORDER, NT, U>, dim3(blocks), dim3(kThreads), st, p);
}

// Up to N = 8 a thread holds all N operands of U vectors in registers (N*U
// at most 16 vectors of 16 bytes); from N = 9 on it streams one vector's
// operands at a time.
template <int N> constexpr int slots_for() { return N <= 4 ? 4 : (N <= 8 ? 2 : 1); }

// Recursive halving, and the tree orders at a power of two: N = 2, 4, ..., 64.
template <class T, class Op, int ORDER>
cudaError_t launch_pow2(const ReduceParams& p, bool rs, cudaStream_t st) {
    switch (p.n) {
    case 2: return launch_one<T, Op, ORDER, 2, slots_for<2>()>(p, rs, st);
    case 4: return launch_one<T, Op, ORDER, 4, slots_for<4>()>(p, rs, st);
    case 8: return launch_one<T, Op, ORDER, 8, slots_for<8>()>(p, rs, st);
    case 16: return launch_one<T, Op, ORDER, 16, 1>(p, rs, st);
    case 32: return launch_one<T, Op, ORDER, 32, 1>(p, rs, st);
    case 64: return launch_one<T, Op, ORDER, 64, 1>(p, rs, st);
    default: return cudaErrorInvalidValue;
    }
}

// The tree orders take any N: compile-time N up to 8 and at the powers of
// two; a run-time N inside the 64-rank envelope otherwise (a rank beyond N
// costs one uniform branch per tree node).  Floats only: the integer types
// run every order on the ring's kernels (vc_reduce_dispatch.cu).
template <class T, class Op, int ORDER>
cudaError_t launch_tree(const ReduceParams& p, bool rs, cudaStream_t st) {
    static_assert(std::is_same<typename Traits<T>::Acc, float>::value,
                  "tree instances exist for the float types only");
    switch (p.n) {
    case 3: return launch_one<T, Op, ORDER, 3, slots_for<3>()>(p, rs, st);
    case 5: return launch_one<T, Op, ORDER, 5, slots_for<5>()>(p, rs, st);
    case 6: return launch_one<T, Op, ORDER, 6, slots_for<6>()>(p, rs, st);
    case 7: return launch_one<T, Op, ORDER, 7, slots_for<7>()>(p, rs, st);
    default:
        if (p.n < 2 || p.n > 64) return cudaErrorInvalidValue;
        if (is_pow2(p.n)) return launch_pow2<T, Op, ORDER>(p, rs, st);
        return launch_one<T, Op, ORDER, -64, 1>(p, rs, st);
    }
}

// The ring takes any N: compile-time N up to 8 and for 16, 32, 64; a
// run-time N otherwise.
template <class T, class Op>
cudaError_t launch_ring(const ReduceParams& p, bool rs, cudaStream_t st) {
    constexpr int R = kOrderRing;
    switch (p.n) {
    case 1: return launch_one<T, Op, R, 1, slots_for<1>()>(p, rs, st);
    case 2: return launch_one<T, Op, R, 2, slots_for<2>()>(p, rs, st);
    case 3: return launch_one<T, Op, R, 3, slots_for<3>()>(p, rs, st);
    case 4: return launch_one<T, Op, R, 4, slots_for<4>()>(p, rs, st);
    case 5: return launch_one<T, Op, R, 5, slots_for<5>()>(p, rs, st);
    case 6: return launch_one<T, Op, R, 6, slots_for<6>()>(p, rs, st);
    case 7: return launch_one<T, Op, R, 7, slots_for<7>()>(p, rs, st);
    case 8: return launch_one<T, Op, R, 8, slots_for<8>()>(p, rs, st);
    case 16: return launch_one<T, Op, R, 16, 1>(p, rs, st);
    case 32: return launch_one<T, Op, R, 32, 1>(p, rs, st);
    case 64: return launch_one<T, Op, R, 64, 1>(p, rs, st);
    default: return launch_one<T, Op, R, 0, 1>(p, rs, st);
    }
}

// The slice of the instances one translation unit holds (the build splits
// them so the units compile in parallel): ring and recursive halving (and
// every order at N = 1, a copy), the tree, or the double binary tree.
enum { kGroupRingRh = 0, kGroupTree = 1, kGroupDoubleTree = 2 };

__host__ __device__ constexpr int order_group(int order, int n) {
    return (n == 1 || order == kOrderRing || order == kOrderRecursiveHalving)
               ? kGroupRingRh
               : (order == kOrderPairwiseTree ? kGroupTree : kGroupDoubleTree);
}

template <class T, class Op, int GROUP>
cudaError_t launch_group(const ReduceParams& p, int order, bool rs, cudaStream_t st) {
    if constexpr (GROUP == kGroupRingRh) {
        // With one rank every order is the identity fold: a copy.  Integers
        // give the same bits in every order, so they only have the ring.
        constexpr bool kInt = !std::is_same<typename Traits<T>::Acc, float>::value;
        if (kInt || p.n == 1 || order == kOrderRing) return launch_ring<T, Op>(p, rs, st);
        if constexpr (!kInt) return launch_pow2<T, Op, kOrderRecursiveHalving>(p, rs, st);
        return cudaErrorInvalidValue;
    } else if constexpr (GROUP == kGroupTree) {
        return launch_tree<T, Op, kOrderPairwiseTree>(p, rs, st);
    } else {
        return launch_tree<T, Op, kOrderDoubleTree>(p, rs, st);
    }
}

}  // namespace vc
