// Dispatch from run-time (op, order, N) to a kernel instance.  Included once
// per element type (vc_reduce_<type>.cu) so the instances compile in
// parallel.
#pragma once

#include "vc_device.cuh"

namespace vc {

template <class T, class Op, int ORDER, int NT>
cudaError_t launch_one(const ReduceParams& p, bool rs, cudaStream_t st) {
    constexpr int V = Traits<T>::V;
    const long long nvec = (p.limit + V - 1) / V;
    if (rs) {
        const int blocks = grid_blocks((const void*)vc_rs_kernel<T, Op, ORDER, NT>, nvec);
        if (blocks < 1) return cudaErrorInvalidConfiguration;
        vc_rs_kernel<T, Op, ORDER, NT><<<blocks, kThreads, 0, st>>>(p);
    } else {
        const int blocks = grid_blocks((const void*)vc_ar_kernel<T, Op, ORDER, NT>, nvec);
        if (blocks < 1) return cudaErrorInvalidConfiguration;
        vc_ar_kernel<T, Op, ORDER, NT><<<blocks, kThreads, 0, st>>>(p);
    }
    return cudaGetLastError();
}

// Recursive halving and the tree are unrolled for N = 2, 4, ..., 64.
template <class T, class Op, int ORDER>
cudaError_t launch_pow2(const ReduceParams& p, bool rs, cudaStream_t st) {
    switch (p.n) {
    case 2: return launch_one<T, Op, ORDER, 2>(p, rs, st);
    case 4: return launch_one<T, Op, ORDER, 4>(p, rs, st);
    case 8: return launch_one<T, Op, ORDER, 8>(p, rs, st);
    case 16: return launch_one<T, Op, ORDER, 16>(p, rs, st);
    case 32: return launch_one<T, Op, ORDER, 32>(p, rs, st);
    case 64: return launch_one<T, Op, ORDER, 64>(p, rs, st);
    default: return cudaErrorInvalidValue;
    }
}

template <class T, class Op>
cudaError_t launch_order(const ReduceParams& p, int order, bool rs, cudaStream_t st) {
    // With one rank every order is the identity fold: a copy.
    if (p.n == 1 || order == kOrderRing) return launch_one<T, Op, kOrderRing, 0>(p, rs, st);
    if (order == kOrderRecursiveHalving)
        return launch_pow2<T, Op, kOrderRecursiveHalving>(p, rs, st);
    return launch_pow2<T, Op, kOrderPairwiseTree>(p, rs, st);
}

// op: 0 sum, 1 prod, 2 max, 3 min, 4 avg (the sum kernel with p.avg set)
template <class T>
cudaError_t launch_reduce_t(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st) {
    switch (op) {
    case 0:
    case 4: return launch_order<T, OpSum>(p, order, rs, st);
    case 1: return launch_order<T, OpProd>(p, order, rs, st);
    case 2: return launch_order<T, OpMax>(p, order, rs, st);
    case 3: return launch_order<T, OpMin>(p, order, rs, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vc
