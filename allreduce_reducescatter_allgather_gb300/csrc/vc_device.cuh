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
constexpr int kGroup = 16;     // loads a streaming fold issues before folding them
constexpr int kRingGroup = 8;  // the same for the ring with a run-time N (whose
                               // run-time rank indices cost more registers)
constexpr int kWaves = 64;  // grid = up to 64 blocks per SM: many more than resident

enum { kOrderRing = 0, kOrderRecursiveHalving = 1, kOrderPairwiseTree = 2, kOrderDoubleTree = 3 };

// Kernel parameters of ReduceScatter / AllReduce.  Passed by value as a
// __grid_constant__ argument, so the pointer tables live in the parameter
// bank and a rank index computed at run time reads them directly.
struct ReduceParams {
    const void* in[kMaxRanks];
    void* out[kMaxRanks];
    long long M;      // logical elements per rank
    long long q;      // shard length ceil(M / N)
    long long limit;  // index space: N*q for ReduceScatter, M for AllReduce
    long long half;   // double binary tree: elements below ceil(M/2) use tree A
    float inv_q;      // 1/q, for the chunk estimate
    int n;            // ranks
    int nout;         // outputs the AllReduce kernel writes: n (AllReduce) or 1 (Reduce)
    int avg;          // divide the sum by n (AVG)
    int vec_ok;       // every base the vector path touches is 16-byte aligned
};

// AllGather, and Broadcast as an AllGather of one shard of q = M elements.
struct GatherParams {
    const void* in[kMaxRanks];  // shards, q elements each
    void* out[kMaxRanks];       // outputs, M elements each
    long long M;
    long long q;
    float inv_q;
    int n;       // outputs written (and shards read, for AllGather)
    int vec_ok;  // every output base 16-byte aligned
    int rpg;     // outputs per rank group: block row y writes outputs
                 // [y*rpg, min(n, (y+1)*rpg)) (more rows when M alone is too
                 // small to fill the GPU)
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

// 16-byte accesses with the default cache policy (measured faster on GB300
// than the evict-first streaming hints for these access patterns).
__device__ __forceinline__ uint4 ld16(const void* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

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

// A loader hands the folds one operand at a time: raw(r) fetches rank r's
// operand in storage form (a 16-byte vector, or one element) and cvt()
// widens it to accumulator lanes.  The folds fetch a whole group with raw()
// before widening any of it, so the group's loads are in flight together
// and only the narrow storage form occupies registers meanwhile.

// The 16-byte vector at element offset i0 of rank r.
template <class T> struct VecLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int W = Traits<T>::V;
    using Raw = uint4;
    const ReduceParams& p;
    long long i0;
    __device__ __forceinline__ Raw raw(int r) const {
        return ld16(static_cast<const T*>(p.in[r]) + i0);
    }
    __device__ __forceinline__ Vec<A, W> cvt(const Raw& u) const {
        Vec<A, W> v;
        unpack(u, v, (T*)nullptr);
        return v;
    }
};

// One element of the padded logical buffer: x^(r)_i below M, the identity
// from M to N*q.
template <class T, class Op> struct ScalarLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int W = 1;
    using Raw = A;
    const ReduceParams& p;
    long long i;
    __device__ __forceinline__ Raw raw(int r) const {
        return (i < p.M) ? load1(static_cast<const T*>(p.in[r]) + i) : Identity<T, Op>::get();
    }
    __device__ __forceinline__ Vec<A, 1> cvt(const Raw& a) const {
        Vec<A, 1> v;
        v.x[0] = a;
        return v;
    }
};

// The 16-byte vector at element offset i0 of rank r, with the rank's base
// pointer taken from a copy of the pointer table in shared memory (for folds
// whose rank index is only known at run time).
template <class T> struct SharedTableLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int W = Traits<T>::V;
    using Raw = uint4;
    const void* const* table;
    long long i0;
    __device__ __forceinline__ Raw raw(int r) const {
        return ld16(static_cast<const T*>(table[r]) + i0);
    }
    __device__ __forceinline__ Vec<A, W> cvt(const Raw& u) const {
        Vec<A, W> v;
        unpack(u, v, (T*)nullptr);
        return v;
    }
};

// Vectors already loaded into registers: buf[r][u] is rank r's vector for
// the thread's slot u.
template <class T, int NR, int U> struct PreLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int W = Traits<T>::V;
    using Raw = uint4;
    const uint4 (&buf)[NR][U];
    int u;
    __device__ __forceinline__ Raw raw(int r) const { return buf[r][u]; }
    __device__ __forceinline__ Vec<A, W> cvt(const Raw& x) const {
        Vec<A, W> v;
        unpack(x, v, (T*)nullptr);
        return v;
    }
};

template <class L> using VecOf = Vec<typename L::A, L::W>;

// The second tree of a double binary tree: node k is played by rank
// (k + 1) mod N, so every rank index stays a compile-time constant.
template <class L, int N> struct ShiftedByOne {
    using A = typename L::A;
    static constexpr int W = L::W;
    using Raw = typename L::Raw;
    const L& l;
    __device__ __forceinline__ Raw raw(int k) const { return l.raw((k + 1) % N); }
    __device__ __forceinline__ Vec<A, W> cvt(const Raw& r) const { return l.cvt(r); }
};

// --------------------------------------------------------------- orders --

// Ring: chunk c is started by rank c and every later rank on the ring adds
// its operand, so the value is the left fold over ranks c, c+1, ..., c+N-1
// (mod N).  Ranks are visited in groups (kGroup with a compile-time N,
// kRingGroup otherwise) whose loads are all issued before any is folded.
template <class Op, int NS, class L>
__device__ __forceinline__ VecOf<L> fold_ring(const L& ld, int n_rt, int c) {
    const int n = NS > 0 ? NS : n_rt;  // NS > 0: N known at compile time
    constexpr int G = NS > 0 ? kGroup : kRingGroup;
    VecOf<L> acc;
    int r = c;
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += G) {
        typename L::Raw t[G];
#pragma unroll
        for (int u = 0; u < G; ++u) {
            if (k0 + u < n) t[u] = ld.raw(r);
            r = (r + 1 == n) ? 0 : r + 1;
        }
        if (k0 == 0) acc = ld.cvt(t[0]);
#pragma unroll
        for (int u = 0; u < G; ++u)
            if (k0 + u < n && k0 + u > 0) acc = vop<Op>(acc, ld.cvt(t[u]));
    }
    return acc;
}

// Recursive halving: the value over ranks {BASE + k*STRIDE : k < CNT} is the
// value over the even k combined with the value over the odd k (the pairing
// at distance N/2 happens first, so it sits at the bottom of the tree).
template <class Op, int KB, int KS, int KC, class L, class R, int G>
__device__ __forceinline__ VecOf<L> rh_local(const L& ld, const R (&t)[G]) {
    if constexpr (KC == 1) {
        return ld.cvt(t[KB]);
    } else {
        return vop<Op>(rh_local<Op, KB, 2 * KS, KC / 2>(ld, t),
                       rh_local<Op, KB + KS, 2 * KS, KC / 2>(ld, t));
    }
}

template <class Op, int BASE, int STRIDE, int CNT, class L>
__device__ __forceinline__ VecOf<L> rh_group(const L& ld) {
    if constexpr (CNT <= kGroup) {
        typename L::Raw t[CNT];
#pragma unroll
        for (int k = 0; k < CNT; ++k) t[k] = ld.raw(BASE + k * STRIDE);
        return rh_local<Op, 0, 1, CNT>(ld, t);
    } else {
        VecOf<L> lo = rh_group<Op, BASE, 2 * STRIDE, CNT / 2>(ld);
        VecOf<L> hi = rh_group<Op, BASE + STRIDE, 2 * STRIDE, CNT / 2>(ld);
        return vop<Op>(lo, hi);
    }
}

// Tree: node P at level L (its lowest set bit) has children P - L/2 and
// P + L/2; its subtree holds ranks P-L+1 .. P+L-1 and its value is
// (left (+) right) (+) own.  Subtrees of at most 15 ranks are loaded as one
// group; t[K] holds rank P-L+1+K.
template <class Op, int K, int L, class Ld, class R, int G>
__device__ __forceinline__ VecOf<Ld> tree_local(const Ld& ld, const R (&t)[G]) {
    if constexpr (L == 1) {
        return ld.cvt(t[K]);
    } else {
        VecOf<Ld> kids = vop<Op>(tree_local<Op, K - L / 2, L / 2>(ld, t),
                                 tree_local<Op, K + L / 2, L / 2>(ld, t));
        return vop<Op>(kids, ld.cvt(t[K]));
    }
}

template <class Op, int P, int L, class Ld>
__device__ __forceinline__ VecOf<Ld> tree_node(const Ld& ld) {
    if constexpr (L == 1) {
        return ld.cvt(ld.raw(P));
    } else if constexpr (2 * L - 1 <= kGroup) {
        typename Ld::Raw t[2 * L - 1];
#pragma unroll
        for (int k = 0; k < 2 * L - 1; ++k) t[k] = ld.raw(P - L + 1 + k);
        return tree_local<Op, L - 1, L>(ld, t);
    } else {
        // the node's own operand is fetched first, so its load is in flight
        // with the subtrees' loads (the combine order is unchanged)
        const typename Ld::Raw own = ld.raw(P);
        VecOf<Ld> l = tree_node<Op, P - L / 2, L / 2>(ld);
        VecOf<Ld> r = tree_node<Op, P + L / 2, L / 2>(ld);
        return vop<Op>(vop<Op>(l, r), ld.cvt(own));
    }
}

// Trees over 16 or more ranks are read in blocks of 16 consecutive ranks.
// Block b holds the whole subtree of node 16b+8 (ranks 16b+1 .. 16b+15) and
// the operand of rank 16b, a node of level 16 or more.  The nodes above the
// blocks are evaluated eagerly in post-order, so only a few partial results
// are live at a time; each block hands its first rank's operand up to the
// node that consumes it.
template <class Op, int B, class Ld>
__device__ __forceinline__ VecOf<Ld> tree_block(const Ld& ld, typename Ld::Raw& first) {
    typename Ld::Raw t[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) t[k] = ld.raw(16 * B + k);
    first = t[0];
    return tree_local<Op, 8, 8>(ld, t);  // t[k] holds rank 16B + k
}

// T(P) for a node of level L >= 8.  `first` receives the operand of the
// lowest rank the subtree's blocks cover, P - L (a node above this one).
// The right child's blocks start at rank P itself, so the operand they hand
// back is this node's own.
template <class Op, int P, int L, class Ld>
__device__ __forceinline__ VecOf<Ld> tree_upper(const Ld& ld, typename Ld::Raw& first) {
    if constexpr (L == 8) {
        return tree_block<Op, (P - 8) / 16>(ld, first);
    } else {
        typename Ld::Raw own;
        VecOf<Ld> l = tree_upper<Op, P - L / 2, L / 2>(ld, first);
        VecOf<Ld> r = tree_upper<Op, P + L / 2, L / 2>(ld, own);
        return vop<Op>(vop<Op>(l, r), ld.cvt(own));
    }
}

// The root, rank 0, has the single child N/2.
template <class Op, int N, class Ld>
__device__ __forceinline__ VecOf<Ld> fold_tree(const Ld& ld) {
    if constexpr (N == 1) {
        return ld.cvt(ld.raw(0));
    } else if constexpr (N >= 16) {
        typename Ld::Raw own0;
        VecOf<Ld> t = tree_upper<Op, N / 2, N / 2>(ld, own0);
        return vop<Op>(t, ld.cvt(own0));
    } else {
        const typename Ld::Raw own = ld.raw(0);
        return vop<Op>(tree_node<Op, N / 2, N / 2>(ld), ld.cvt(own));
    }
}

// Ring with N known at compile time: the left fold starting at rank C, with
// every rank index a constant (operands may already sit in registers).
template <class Op, int N, int C, class L>
__device__ __forceinline__ VecOf<L> ring_from(const L& ld) {
    VecOf<L> acc = ld.cvt(ld.raw(C));
#pragma unroll
    for (int k = 1; k < N; ++k) acc = vop<Op>(acc, ld.cvt(ld.raw((C + k) % N)));
    return acc;
}

// Picks the rotation for chunk c among the N compile-time ones.
template <class Op, int N, int C, class L>
__device__ __forceinline__ VecOf<L> ring_switch(const L& ld, int c) {
    if constexpr (C == N - 1) {
        return ring_from<Op, N, C>(ld);
    } else {
        if (c == C) return ring_from<Op, N, C>(ld);
        return ring_switch<Op, N, C + 1>(ld, c);
    }
}

// NT > 0: N is a compile-time constant; NT == 0: ring with a run-time N.
// The ring switches among its rotations up to N = 8 and folds in groups
// with run-time rank indices beyond.  `sel` is the ring's chunk, or for the
// double binary tree which tree (0 = A, 1 = B) the element belongs to.
template <class Op, int ORDER, int NT, class L>
__device__ __forceinline__ VecOf<L> fold(const L& ld, int n, int sel) {
    const int c = sel;
    if constexpr (ORDER == kOrderRecursiveHalving) {
        return rh_group<Op, 0, 1, NT>(ld);
    } else if constexpr (ORDER == kOrderPairwiseTree) {
        return fold_tree<Op, NT>(ld);
    } else if constexpr (ORDER == kOrderDoubleTree) {
        if (sel == 0) return fold_tree<Op, NT>(ld);
        ShiftedByOne<L, NT> shifted{ld};
        return fold_tree<Op, NT>(shifted);
    } else if constexpr (NT > 0 && NT <= 8) {
        return ring_switch<Op, NT, 0>(ld, c);
    } else {
        return fold_ring<Op, NT>(ld, n, c);
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

// The result vector of elements i0 .. i0+V-1 (chunk c) to its destination:
// AllReduce, all N outputs; ReduceScatter, the shard that owns it.
template <class T, int NT, bool RS, class A, int V>
__device__ __forceinline__ void store_result(const ReduceParams& p, int c, long long i0,
                                             Vec<A, V>& acc) {
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
            for (int s = 0; s < NT; ++s)
                if (s < p.nout) st16(static_cast<T*>(p.out[s]) + i0, u);
        } else {
            for (int s = 0; s < p.nout; ++s) st16(static_cast<T*>(p.out[s]) + i0, u);
        }
    }
}

// Reduces one element the slow way (misaligned bases, a vector straddling a
// chunk boundary or the end of the data, or the padding).
template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __noinline__ void reduce_one(const ReduceParams& p, long long i) {
    using A = typename Traits<T>::Acc;
    const int c = chunk_of(i, p.q, p.inv_q, p.n);
    ScalarLoader<T, Op> ld{p, i};
    const int sel = (ORDER == kOrderDoubleTree) ? (i >= p.half) : c;
    Vec<A, 1> v = fold<Op, ORDER, NT>(ld, p.n, sel);
    A r = v.x[0];
    if (p.avg) r = avg_div(r, p.n);
    if constexpr (RS) {
        store1(static_cast<T*>(p.out[c]) + (i - (long long)c * p.q), r);
    } else {
        for (int s = 0; s < p.nout; ++s) store1(static_cast<T*>(p.out[s]) + i, r);
    }
}

// One vector slot on its own: the vector path if it lies inside one chunk
// and inside the data on aligned bases, else element by element.
template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __noinline__ void reduce_slot(const ReduceParams& p, long long v) {
    constexpr int V = Traits<T>::V;
    const long long i0 = v * V;
    const int c = chunk_of(i0, p.q, p.inv_q, p.n);
    const bool one_tree = (ORDER != kOrderDoubleTree) || i0 >= p.half || i0 + V <= p.half;
    if (p.vec_ok && one_tree && i0 + V <= p.M && i0 + V <= (long long)(c + 1) * p.q) {
        VecLoader<T> ld{p, i0};
        const int sel = (ORDER == kOrderDoubleTree) ? (i0 >= p.half) : c;
        auto acc = fold<Op, ORDER, NT>(ld, p.n, sel);
        store_result<T, NT, RS>(p, c, i0, acc);
    } else {
        for (int k = 0; k < V && i0 + k < p.limit; ++k) reduce_one<T, Op, ORDER, NT, RS>(p, i0 + k);
    }
}

// The kernel body.  A block takes U*blockDim.x consecutive vectors per
// iteration; thread t owns the U vectors t, t + blockDim.x, ... of that
// range (each warp access is 512 contiguous bytes).  When all U vectors sit
// inside one chunk and inside the data on aligned bases (nearly always), the
// thread issues every load before it folds or stores anything:
//  - N <= 8 (NT > 0): the N x U vectors (at most 16) are loaded into
//    registers in rank order, with constant rank indices, then folded slot by
//    slot in the order's tree (the ring picks its rotation by the chunk);
//  - otherwise (U = 1): the fold streams its operands in groups of kGroup;
//    the ring with run-time N reads its rotated pointers from shared memory.
// Anything else goes slot by slot through reduce_slot.
template <class T, class Op, int ORDER, int NT, int U, bool RS>
__device__ __forceinline__ void reduce_body(const ReduceParams& p) {
    constexpr int V = Traits<T>::V;
    constexpr bool kPre = (NT > 0 && NT <= 8);
    // ring beyond 8 ranks: rotated rank indices read from shared memory
    constexpr bool kTable = (ORDER == kOrderRing && (NT == 0 || NT > 8));
    __shared__ const void* s_in[kTable ? kMaxRanks : 1];
    __shared__ void* s_out[kTable ? kMaxRanks : 1];
    if constexpr (kTable) {
        for (int r = threadIdx.x; r < p.n; r += blockDim.x) {
            s_in[r] = p.in[r];
            s_out[r] = p.out[r];
        }
        __syncthreads();
    }
    const long long nvec = (p.limit + V - 1) / V;
    const long long span = (long long)blockDim.x * U;
    for (long long b0 = (long long)blockIdx.x * span; b0 < nvec; b0 += (long long)gridDim.x * span) {
        const long long v0 = b0 + threadIdx.x;
        const long long vlast = v0 + (long long)(U - 1) * blockDim.x;
        bool wide = false;
        int c = 0;
        if (vlast < nvec && p.vec_ok) {
            c = chunk_of(v0 * V, p.q, p.inv_q, p.n);
            const long long end = vlast * V + V;
            wide = end <= p.M && end <= (long long)(c + 1) * p.q;
            if constexpr (ORDER == kOrderDoubleTree)
                wide = wide && (v0 * V >= p.half || end <= p.half);
        }
        // the fold's selector: the ring's chunk, or the double tree's half
        const int sel = (ORDER == kOrderDoubleTree) ? (int)(v0 * V >= p.half) : c;
        if (wide) {
            if constexpr (kPre) {
                uint4 buf[NT][U];
#pragma unroll
                for (int r = 0; r < NT; ++r) {
                    const T* base = static_cast<const T*>(p.in[r]) + v0 * V;
#pragma unroll
                    for (int u = 0; u < U; ++u) buf[r][u] = ld16(base + (long long)u * blockDim.x * V);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    PreLoader<T, NT, U> ld{buf, u};
                    auto acc = fold<Op, ORDER, NT>(ld, NT, sel);
                    store_result<T, NT, RS>(p, c, (v0 + (long long)u * blockDim.x) * V, acc);
                }
            } else if constexpr (kTable) {
                static_assert(U == 1, "streaming folds take one vector per thread");
                SharedTableLoader<T> ld{s_in, v0 * V};
                auto acc = fold<Op, ORDER, NT>(ld, p.n, c);
                if (p.avg) {
#pragma unroll
                    for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
                }
                const long long i0 = v0 * V;
                if constexpr (RS) {
                    T* dst = static_cast<T*>(s_out[c]) + (i0 - (long long)c * p.q);
                    if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                        st16(dst, pack(acc, (T*)nullptr));
                    } else {
#pragma unroll
                        for (int k = 0; k < V; ++k) store1(dst + k, acc.x[k]);
                    }
                } else {
                    const uint4 u = pack(acc, (T*)nullptr);
                    for (int s = 0; s < p.nout; ++s) st16(static_cast<T*>(s_out[s]) + i0, u);
                }
            } else {
                static_assert(U == 1, "streaming folds take one vector per thread");
                VecLoader<T> ld{p, v0 * V};
                auto acc = fold<Op, ORDER, NT>(ld, p.n, sel);
                store_result<T, NT, RS>(p, c, v0 * V, acc);
            }
        } else {
#pragma unroll 1
            for (int u = 0; u < U; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) reduce_slot<T, Op, ORDER, NT, RS>(p, v);
            }
        }
    }
    // This block is done: a kernel launched after this one with programmatic
    // stream serialization may start now (it waits for the whole grid, and
    // for its memory, before it touches any; see vc_ag_kernel).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ReduceScatter: index space [0, N*q), one store per element into the shard
// that owns it.
// Both reduction kernels state "at least one resident block" explicitly.
// Measured on GB300 against the bare launch bound: ptxas then keeps more
// loads in flight per thread, which lifts AllReduce by 0.5-1 % across the
// board and the 64-rank tree from 0.78x to 1.06x the copy rate (the one
// loss measured: bf16 RS at 32 ranks in the tree orders, 7.19 -> 6.54 TB/s).
template <class T, class Op, int ORDER, int NT, int U>
__global__ void __launch_bounds__(kThreads, 1) vc_rs_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, U, true>(p);
}

// Fused AllReduce: index space [0, M), N stores per element (one, to the
// root's buffer, for Reduce).
template <class T, class Op, int ORDER, int NT, int U>
__global__ void __launch_bounds__(kThreads, 1) vc_ar_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, U, false>(p);
}

// AllGather: output index i comes from shard s = floor(i/q) at offset i - sq,
// and is written to all N outputs.  It moves bits only, so it is typed by
// element size alone.  Like the reductions, a thread takes kGatherSlots
// vectors (blockDim.x apart) and loads all of them before it stores any.
// When the M output indices alone give too few blocks for the GPU (small M,
// many ranks), the outputs are split into groups along the grid's y axis:
// each group re-reads the (small) source and writes its share of the ranks.
template <int ES> struct Bits;
template <> struct Bits<2> { using U = unsigned short; };
template <> struct Bits<4> { using U = unsigned; };
template <> struct Bits<8> { using U = unsigned long long; };

constexpr int kGatherSlots = 8;

template <int ES>
__device__ __forceinline__ uint4 gather_load(const GatherParams& p, int s, long long i0) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
    const U* src = static_cast<const U*>(p.in[s]) + (i0 - (long long)s * p.q);
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) return ld16(src);
    union {
        U t[V];
        uint4 u;
    } w;
#pragma unroll
    for (int k = 0; k < V; ++k) w.t[k] = src[k];
    return w.u;
}

template <int ES>
__device__ __noinline__ void gather_slot(const GatherParams& p, long long v, int r0, int r1) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
    const long long i0 = v * V;
    const int s = chunk_of(i0, p.q, p.inv_q, p.n);
    if (p.vec_ok && i0 + V <= p.M && i0 + V <= (long long)(s + 1) * p.q) {
        const uint4 val = gather_load<ES>(p, s, i0);
        for (int r = r0; r < r1; ++r) st16(static_cast<U*>(p.out[r]) + i0, val);
    } else {
        for (int k = 0; k < V && i0 + k < p.M; ++k) {
            const long long i = i0 + k;
            const int si = chunk_of(i, p.q, p.inv_q, p.n);
            const U val = static_cast<const U*>(p.in[si])[i - (long long)si * p.q];
            for (int r = r0; r < r1; ++r) static_cast<U*>(p.out[r])[i] = val;
        }
    }
}

template <int ES>
__global__ void __launch_bounds__(kThreads) vc_ag_kernel(const __grid_constant__ GatherParams p) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
    constexpr int S = kGatherSlots;
    // Launched with programmatic stream serialization, this grid may begin
    // while the kernel before it (the ReduceScatter of a decomposed
    // AllReduce) finishes; wait for that grid to complete and its writes to
    // be visible before the first access to global memory.  (Launched
    // normally, or after a kernel that never signals, this returns at once
    // or when that kernel has completed.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long nvec = (p.M + V - 1) / V;
    const long long span = (long long)blockDim.x * S;
    const int r0 = (int)blockIdx.y * p.rpg;
    const int r1 = min(p.n, r0 + p.rpg);
    for (long long b0 = (long long)blockIdx.x * span; b0 < nvec; b0 += (long long)gridDim.x * span) {
        const long long v0 = b0 + threadIdx.x;
        const long long vlast = v0 + (long long)(S - 1) * blockDim.x;
        bool wide = false;
        int s = 0;
        if (vlast < nvec && p.vec_ok) {
            s = chunk_of(v0 * V, p.q, p.inv_q, p.n);
            const long long end = vlast * V + V;
            wide = end <= p.M && end <= (long long)(s + 1) * p.q;
        }
        if (wide) {
            uint4 val[S];
#pragma unroll
            for (int u = 0; u < S; ++u) val[u] = gather_load<ES>(p, s, (v0 + (long long)u * blockDim.x) * V);
            for (int r = r0; r < r1; ++r) {
                U* dst = static_cast<U*>(p.out[r]) + v0 * V;
#pragma unroll
                for (int u = 0; u < S; ++u) st16(dst + (long long)u * blockDim.x * V, val[u]);
            }
        } else {
#pragma unroll 1
            for (int u = 0; u < S; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) gather_slot<ES>(p, v, r0, r1);
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

// Blocks for a grid-stride kernel over `units` thread-units: enough for
// every unit, at most kWaves blocks per SM.  (Many more blocks than fit at
// once keep the blocks in flight on neighbouring addresses, which the HBM
// serves faster than one resident wave striding over the whole buffer.)
int grid_blocks(long long units);

// SMs of the current device (queried once per device); -1 on error.
int sm_count();

}  // namespace vc
