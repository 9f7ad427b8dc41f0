// Device-side building blocks of the virtual-rank collectives: element types,
// reduction ops, the three reduction orders as register folds, and the kernels.
//
// Every output element depends only on the N operands at the same index, so
// a thread owns a 16-byte vector of consecutive indices, loads it from each
// of the N rank buffers, folds the N vectors lane by lane in the order's fixed
// tree, and stores the result (AllReduce: to all N outputs; ReduceScatter: to
// the shard that owns the index).  Nothing waits on anything: no barrier, no
// flag, no inter-block traffic.  The work is bound by HBM bandwidth, so the
// design is about keeping many 16-byte loads in flight (groups of up to 8
// independent loads per thread, a grid of whole waves of resident blocks) and
// about never re-reading a byte.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace vc {

constexpr int kMaxRanks = 64;
constexpr int kThreads = 256;
constexpr int kGroup = 8;  // loads issued together before they are folded

enum { kOrderRing = 0, kOrderRecursiveHalving = 1, kOrderPairwiseTree = 2 };

// Kernel parameters of ReduceScatter / AllReduce.  Passed by value as a
// __grid_constant__ argument, so the pointer tables live in the parameter
// bank and a rank index computed at run time reads them directly.
struct ReduceParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    long long M;      // logical elements per rank
    long long q;      // shard length ceil(M / N)
    long long limit;  // index space: N*q for ReduceScatter, M for AllReduce
    float inv_q;      // 1/q, for the chunk estimate
    int n;            // ranks
    int avg;          // divide the sum by n (AVG)
    int vec_ok;       // every base the vector path touches is 16-byte aligned
};

struct GatherParams {
    const void* in[kMaxRanks];  // shards, q elements each
    void* out[kMaxRanks];       // outputs, M elements each
    long long M;
    long long q;
    float inv_q;
    int n;
    int vec_ok;  // every output base 16-byte aligned
};

// ---------------------------------------------------------------- types --

template <class T> struct Traits;
template <> struct Traits<int32_t> {
    using Acc = long long;  // 64-bit accumulation, wraps; low 32 bits stored
    static constexpr int V = 4;
};
template <> struct Traits<long long> {
    using Acc = long long;
    static constexpr int V = 2;
};
template <> struct Traits<float> {
    using Acc = float;
    static constexpr int V = 4;
};
template <> struct Traits<__nv_bfloat16> {
    using Acc = float;  // widened exactly; rounded once at the store
    static constexpr int V = 8;
};

template <class A, int W> struct Vec {
    A x[W];
};

// 16 bytes -> V accumulator lanes (little-endian lane order).
__device__ __forceinline__ void unpack(const uint4 u, Vec<long long, 4>& a, int32_t*) {
    a.x[0] = (long long)(int32_t)u.x;
    a.x[1] = (long long)(int32_t)u.y;
    a.x[2] = (long long)(int32_t)u.z;
    a.x[3] = (long long)(int32_t)u.w;
}
__device__ __forceinline__ void unpack(const uint4 u, Vec<long long, 2>& a, long long*) {
    a.x[0] = (long long)(((unsigned long long)u.y << 32) | u.x);
    a.x[1] = (long long)(((unsigned long long)u.w << 32) | u.z);
}
__device__ __forceinline__ void unpack(const uint4 u, Vec<float, 4>& a, float*) {
    a.x[0] = __uint_as_float(u.x);
    a.x[1] = __uint_as_float(u.y);
    a.x[2] = __uint_as_float(u.z);
    a.x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4 u, Vec<float, 8>& a, __nv_bfloat16*) {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        a.x[2 * k] = __uint_as_float(w[k] << 16);
        a.x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

// V lanes -> 16 bytes, narrowing to the storage type.
__device__ __forceinline__ uint4 pack(const Vec<long long, 4>& a, int32_t*) {
    return make_uint4((unsigned)(unsigned long long)a.x[0], (unsigned)(unsigned long long)a.x[1],
                      (unsigned)(unsigned long long)a.x[2], (unsigned)(unsigned long long)a.x[3]);
}
__device__ __forceinline__ uint4 pack(const Vec<long long, 2>& a, long long*) {
    const unsigned long long u0 = (unsigned long long)a.x[0], u1 = (unsigned long long)a.x[1];
    return make_uint4((unsigned)u0, (unsigned)(u0 >> 32), (unsigned)u1, (unsigned)(u1 >> 32));
}
__device__ __forceinline__ uint4 pack(const Vec<float, 4>& a, float*) {
    return make_uint4(__float_as_uint(a.x[0]), __float_as_uint(a.x[1]), __float_as_uint(a.x[2]),
                      __float_as_uint(a.x[3]));
}
__device__ __forceinline__ unsigned bf16_bits(float f) {
    return (unsigned)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint4 pack(const Vec<float, 8>& a, __nv_bfloat16*) {
    unsigned w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = bf16_bits(a.x[2 * k]) | (bf16_bits(a.x[2 * k + 1]) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// One element: load widened / store narrowed.
__device__ __forceinline__ long long load1(const int32_t* p) { return (long long)*p; }
__device__ __forceinline__ long long load1(const long long* p) { return *p; }
__device__ __forceinline__ float load1(const float* p) { return *p; }
__device__ __forceinline__ float load1(const __nv_bfloat16* p) {
    return __uint_as_float((unsigned)*reinterpret_cast<const unsigned short*>(p) << 16);
}
__device__ __forceinline__ void store1(int32_t* p, long long v) {
    *p = (int32_t)(unsigned)(unsigned long long)v;
}
__device__ __forceinline__ void store1(long long* p, long long v) { *p = v; }
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }
__device__ __forceinline__ void store1(__nv_bfloat16* p, float v) {
    *reinterpret_cast<unsigned short*>(p) = (unsigned short)bf16_bits(v);
}

// Streaming 16-byte accesses: each byte is touched once, so ask the caches
// to evict it first.
__device__ __forceinline__ uint4 ld16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }

// ------------------------------------------------------------------- ops --

// a (+) b with the running value on the left.  Floats: one IEEE single
// operation, explicitly rounded (no contraction into FMA).  Integers: wrap
// modulo 2^64.  MAX/MIN keep a on ties.
struct OpSum {
    __device__ static __forceinline__ float apply(float a, float b) { return __fadd_rn(a, b); }
    __device__ static __forceinline__ long long apply(long long a, long long b) {
        return (long long)((unsigned long long)a + (unsigned long long)b);
    }
};
struct OpProd {
    __device__ static __forceinline__ float apply(float a, float b) { return __fmul_rn(a, b); }
    __device__ static __forceinline__ long long apply(long long a, long long b) {
        return (long long)((unsigned long long)a * (unsigned long long)b);
    }
};
struct OpMax {
    template <class A> __device__ static __forceinline__ A apply(A a, A b) { return b > a ? b : a; }
};
struct OpMin {
    template <class A> __device__ static __forceinline__ A apply(A a, A b) { return b < a ? b : a; }
};

// The padding value e(op, T) in the accumulator domain.
template <class T, class Op> struct Identity;
template <class T> struct Identity<T, OpSum> {
    __device__ static __forceinline__ typename Traits<T>::Acc get() { return 0; }
};
template <class T> struct Identity<T, OpProd> {
    __device__ static __forceinline__ typename Traits<T>::Acc get() { return 1; }
};
template <> struct Identity<int32_t, OpMax> {
    __device__ static __forceinline__ long long get() { return -2147483647LL - 1; }
};
template <> struct Identity<int32_t, OpMin> {
    __device__ static __forceinline__ long long get() { return 2147483647LL; }
};
template <> struct Identity<long long, OpMax> {
    __device__ static __forceinline__ long long get() { return (long long)(1ULL << 63); }
};
template <> struct Identity<long long, OpMin> {
    __device__ static __forceinline__ long long get() { return (long long)((1ULL << 63) - 1); }
};
template <class T> struct IdentityF {
    __device__ static __forceinline__ float neg_inf() { return __uint_as_float(0xff800000u); }
    __device__ static __forceinline__ float pos_inf() { return __uint_as_float(0x7f800000u); }
};
template <> struct Identity<float, OpMax> {
    __device__ static __forceinline__ float get() { return IdentityF<float>::neg_inf(); }
};
template <> struct Identity<float, OpMin> {
    __device__ static __forceinline__ float get() { return IdentityF<float>::pos_inf(); }
};
template <> struct Identity<__nv_bfloat16, OpMax> {
    __device__ static __forceinline__ float get() { return IdentityF<float>::neg_inf(); }
};
template <> struct Identity<__nv_bfloat16, OpMin> {
    __device__ static __forceinline__ float get() { return IdentityF<float>::pos_inf(); }
};

template <class Op, class A, int W>
__device__ __forceinline__ Vec<A, W> vop(const Vec<A, W>& a, const Vec<A, W>& b) {
    Vec<A, W> r;
#pragma unroll
    for (int k = 0; k < W; ++k) r.x[k] = Op::apply(a.x[k], b.x[k]);
    return r;
}

// AVG: one division by n after the ordered sum.
__device__ __forceinline__ float avg_div(float s, int n) { return __fdiv_rn(s, (float)n); }
__device__ __forceinline__ long long avg_div(long long s, int n) { return s / (long long)n; }

// ------------------------------------------------------------- loaders --

// Loads the 16-byte vector at element offset i0 of rank r.
template <class T> struct VecLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int V = Traits<T>::V;
    const ReduceParams& p;
    long long i0;
    __device__ __forceinline__ Vec<A, V> operator()(int r) const {
        Vec<A, V> v;
        unpack(ld16(static_cast<const T*>(p.in[r]) + i0), v, (T*)nullptr);
        return v;
    }
};

// Loads one element of the padded logical buffer: x^(r)_i below M, the
// identity from M to N*q.
template <class T, class Op> struct ScalarLoader {
    using A = typename Traits<T>::Acc;
    const ReduceParams& p;
    long long i;
    __device__ __forceinline__ Vec<A, 1> operator()(int r) const {
        Vec<A, 1> v;
        v.x[0] = (i < p.M) ? load1(static_cast<const T*>(p.in[r]) + i) : Identity<T, Op>::get();
        return v;
    }
};

// --------------------------------------------------------------- orders --

// Ring: chunk c is started by rank c and every later rank on the ring adds
// its operand, so the value is the left fold over ranks c, c+1, ..., c+N-1
// (mod N).  Ranks are visited in groups of kGroup whose loads are all issued
// before any of them is folded.
template <class Op, class A, int W, class L>
__device__ __forceinline__ Vec<A, W> fold_ring(const L& ld, int n, int c) {
    Vec<A, W> acc;
    int r = c;
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += kGroup) {
        Vec<A, W> t[kGroup];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
            if (k0 + u < n) t[u] = ld(r);
            r = (r + 1 == n) ? 0 : r + 1;
        }
        if (k0 == 0) acc = t[0];
#pragma unroll
        for (int u = 0; u < kGroup; ++u)
            if (k0 + u < n && k0 + u > 0) acc = vop<Op>(acc, t[u]);
    }
    return acc;
}

// Recursive halving: the value over ranks {BASE + k*STRIDE : k < CNT} is the
// value over the even k combined with the value over the odd k (the pairing
// at distance N/2 happens first, so it sits at the bottom of the tree).
template <class Op, class A, int W, int KB, int KS, int KC, int G>
__device__ __forceinline__ Vec<A, W> rh_local(const Vec<A, W> (&t)[G]) {
    if constexpr (KC == 1) {
        return t[KB];
    } else {
        return vop<Op>(rh_local<Op, A, W, KB, 2 * KS, KC / 2>(t),
                       rh_local<Op, A, W, KB + KS, 2 * KS, KC / 2>(t));
    }
}

template <class Op, class A, int W, int BASE, int STRIDE, int CNT, class L>
__device__ __forceinline__ Vec<A, W> rh_group(const L& ld) {
    if constexpr (CNT <= kGroup) {
        Vec<A, W> t[CNT];
#pragma unroll
        for (int k = 0; k < CNT; ++k) t[k] = ld(BASE + k * STRIDE);
        return rh_local<Op, A, W, 0, 1, CNT>(t);
    } else {
        Vec<A, W> lo = rh_group<Op, A, W, BASE, 2 * STRIDE, CNT / 2>(ld);
        Vec<A, W> hi = rh_group<Op, A, W, BASE + STRIDE, 2 * STRIDE, CNT / 2>(ld);
        return vop<Op>(lo, hi);
    }
}

// Tree: node P at level L (its lowest set bit) has children P - L/2 and
// P + L/2; its subtree holds ranks P-L+1 .. P+L-1 and its value is
// (left (+) right) (+) own.  Subtrees of at most 7 ranks are loaded as one
// group; t[K] holds rank P-L+1+K.
template <class Op, class A, int W, int K, int L, int G>
__device__ __forceinline__ Vec<A, W> tree_local(const Vec<A, W> (&t)[G]) {
    if constexpr (L == 1) {
        return t[K];
    } else {
        Vec<A, W> kids = vop<Op>(tree_local<Op, A, W, K - L / 2, L / 2>(t),
                                 tree_local<Op, A, W, K + L / 2, L / 2>(t));
        return vop<Op>(kids, t[K]);
    }
}

template <class Op, class A, int W, int P, int L, class Ld>
__device__ __forceinline__ Vec<A, W> tree_node(const Ld& ld) {
    if constexpr (L == 1) {
        return ld(P);
    } else if constexpr (L <= 4) {
        Vec<A, W> t[2 * L - 1];
#pragma unroll
        for (int k = 0; k < 2 * L - 1; ++k) t[k] = ld(P - L + 1 + k);
        return tree_local<Op, A, W, L - 1, L>(t);
    } else {
        Vec<A, W> l = tree_node<Op, A, W, P - L / 2, L / 2>(ld);
        Vec<A, W> r = tree_node<Op, A, W, P + L / 2, L / 2>(ld);
        return vop<Op>(vop<Op>(l, r), ld(P));
    }
}

// The root, rank 0, has the single child N/2.
template <class Op, class A, int W, int N, class Ld>
__device__ __forceinline__ Vec<A, W> fold_tree(const Ld& ld) {
    if constexpr (N == 1) {
        return ld(0);
    } else {
        return vop<Op>(tree_node<Op, A, W, N / 2, N / 2>(ld), ld(0));
    }
}

template <class Op, int ORDER, int NT, class A, int W, class L>
__device__ __forceinline__ Vec<A, W> fold(const L& ld, int n, int c) {
    if constexpr (ORDER == kOrderRecursiveHalving) {
        return rh_group<Op, A, W, 0, 1, NT>(ld);
    } else if constexpr (ORDER == kOrderPairwiseTree) {
        return fold_tree<Op, A, W, NT>(ld);
    } else {
        return fold_ring<Op, A, W>(ld, n, c);
    }
}

// --------------------------------------------------------- chunk index --

// c = floor(i / q), from a single-precision estimate corrected by one step.
// The estimate's relative error is a few units of 2^-24 and i/q < 64, so it
// is off by at most one.
__device__ __forceinline__ int chunk_of(long long i, long long q, float inv_q, int n) {
    int c = (int)(__ll2float_rn(i) * inv_q);
    c = c < 0 ? 0 : (c > n - 1 ? n - 1 : c);
    if ((long long)c * q > i)
        --c;
    else if (c + 1 < n && (long long)(c + 1) * q <= i)
        ++c;
    return c;
}

// --------------------------------------------------------------- kernels --

// Reduces one element the slow way (misaligned bases, a vector straddling a
// chunk boundary or the end of the data, or the padding).
template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __noinline__ void reduce_one(const ReduceParams& p, long long i) {
    using A = typename Traits<T>::Acc;
    const int c = chunk_of(i, p.q, p.inv_q, p.n);
    ScalarLoader<T, Op> ld{p, i};
    Vec<A, 1> v = fold<Op, ORDER, NT, A, 1>(ld, p.n, c);
    A r = v.x[0];
    if (p.avg) r = avg_div(r, p.n);
    if constexpr (RS) {
        store1(static_cast<T*>(p.out[c]) + (i - (long long)c * p.q), r);
    } else {
        const int n = NT ? NT : p.n;
        for (int s = 0; s < n; ++s) store1(static_cast<T*>(p.out[s]) + i, r);
    }
}

template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __forceinline__ void reduce_body(const ReduceParams& p) {
    using A = typename Traits<T>::Acc;
    constexpr int V = Traits<T>::V;
    const long long nvec = (p.limit + V - 1) / V;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        const long long i0 = v * V;
        const int c = chunk_of(i0, p.q, p.inv_q, p.n);
        const long long cend = (long long)(c + 1) * p.q;
        if (p.vec_ok && i0 + V <= p.M && i0 + V <= cend) {
            VecLoader<T> ld{p, i0};
            Vec<A, V> acc = fold<Op, ORDER, NT, A, V>(ld, p.n, c);
            if (p.avg) {
#pragma unroll
                for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
            }
            if constexpr (RS) {
                T* dst = static_cast<T*>(p.out[c]) + (i0 - (long long)c * p.q);
                if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                    st16(dst, pack(acc, (T*)nullptr));
                } else {
#pragma unroll
                    for (int k = 0; k < V; ++k) store1(dst + k, acc.x[k]);
                }
            } else {
                const uint4 u = pack(acc, (T*)nullptr);
                if constexpr (NT > 0) {
#pragma unroll
                    for (int s = 0; s < NT; ++s) st16(static_cast<T*>(p.out[s]) + i0, u);
                } else {
                    for (int s = 0; s < p.n; ++s) st16(static_cast<T*>(p.out[s]) + i0, u);
                }
            }
        } else {
            for (int k = 0; k < V && i0 + k < p.limit; ++k)
                reduce_one<T, Op, ORDER, NT, RS>(p, i0 + k);
        }
    }
}

// ReduceScatter: index space [0, N*q), one store per element into the shard
// that owns it.
template <class T, class Op, int ORDER, int NT>
__global__ void __launch_bounds__(kThreads) vc_rs_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, true>(p);
}

// Fused AllReduce: index space [0, M), N stores per element.
template <class T, class Op, int ORDER, int NT>
__global__ void __launch_bounds__(kThreads) vc_ar_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, false>(p);
}

// AllGather: output index i comes from shard s = floor(i/q) at offset i - sq,
// and is written to all N outputs.  It moves bits only, so it is typed by
// element size alone.
template <int ES> struct Bits;
template <> struct Bits<2> { using U = unsigned short; };
template <> struct Bits<4> { using U = unsigned; };
template <> struct Bits<8> { using U = unsigned long long; };

template <int ES>
__global__ void __launch_bounds__(kThreads) vc_ag_kernel(const __grid_constant__ GatherParams p) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
    const long long nvec = (p.M + V - 1) / V;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
        const long long i0 = v * V;
        const int s = chunk_of(i0, p.q, p.inv_q, p.n);
        const long long send = (long long)(s + 1) * p.q;
        if (p.vec_ok && i0 + V <= p.M && i0 + V <= send) {
            const U* src = static_cast<const U*>(p.in[s]) + (i0 - (long long)s * p.q);
            uint4 val;
            if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
                val = ld16(src);
            } else {
                union {
                    U t[V];
                    uint4 u;
                } w;
#pragma unroll
                for (int k = 0; k < V; ++k) w.t[k] = src[k];
                val = w.u;
            }
            for (int r = 0; r < p.n; ++r) st16(static_cast<U*>(p.out[r]) + i0, val);
        } else {
            for (int k = 0; k < V && i0 + k < p.M; ++k) {
                const long long i = i0 + k;
                const int si = chunk_of(i, p.q, p.inv_q, p.n);
                const U val = static_cast<const U*>(p.in[si])[i - (long long)si * p.q];
                for (int r = 0; r < p.n; ++r) static_cast<U*>(p.out[r])[i] = val;
            }
        }
    }
}

// Launchers, one translation unit per element type (vc_reduce_<type>.cu).
cudaError_t launch_reduce_i32(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st);
cudaError_t launch_reduce_i64(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st);
cudaError_t launch_reduce_f32(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st);
cudaError_t launch_reduce_bf16(const ReduceParams& p, int op, int order, bool rs, cudaStream_t st);
cudaError_t launch_gather(const GatherParams& p, int esize, cudaStream_t st);

// Blocks for a grid-stride kernel: enough for every vector, at most one
// full wave of resident blocks on every SM.
int grid_blocks(const void* kernel, long long nvec);

}  // namespace vc
