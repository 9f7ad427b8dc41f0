// Device-side building blocks of the virtual-rank collectives: element types,
// reduction ops, the three reduction orders as register folds, and the kernels.
//
// Every output element depends only on the N operands at the same index, so
// a thread owns a 16-byte vector of consecutive indices, loads it from each
// of the N rank buffers, folds the N vectors lane by lane in the order's fixed
// tree, and stores the result (AllReduce: to all N outputs; ReduceScatter: to
// the shard that owns the index).  No block waits on another: no flag, no
// inter-block traffic.  (The barriers are a block's own __syncthreads after
// it copies the pointer table to shared memory, and the warp-wide shuffles
// of the realigned shard accesses; the one wait is each kernel's grid
// dependency on the kernel before it, which the hardware releases when that
// kernel completes.)  The work is bound by
// HBM bandwidth, so the design is about keeping many 16-byte loads in flight
// (up to 16 independent loads per thread, many more blocks than are
// resident) and about never re-reading a byte.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

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
// Two lanes per conversion (each rounded to nearest even on its own, lane
// 2k in the low half): the bits of two bf16_bits calls, in one instruction.
__device__ __forceinline__ uint4 pack(const Vec<float, 8>& a, __nv_bfloat16*) {
    unsigned w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a.x[2 * k], a.x[2 * k + 1]);
        w[k] = *reinterpret_cast<const unsigned*>(&h);
    }
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

// 16-byte accesses with the default cache policy.  Measured on GB300 with
// the evict-first streaming hints instead: stores cost the AllReduce
// 0.2-0.4 % of the copy rate and loads 1-1.6 %; the ReduceScatter gained
// nothing from either on data that does not stay in L2.
__host__ __device__ __forceinline__ uint4 ld16(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}
__host__ __device__ __forceinline__ void st16(void* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// A 16-byte store with the evict-first streaming hint, for the AllGather's
// N output streams (N >= 4).  Measured on GB300 (back-to-back calls): 0.3-1 %
// of the copy rate at 4 x 256 MiB, 8 x 64 MiB and 8 x 1 GiB, and the
// decomposed AllReduce of a 25 MiB bf16 bucket on 8 ranks 0.93x -> 0.94x
// (the gather's own writes leave L2 first, so the shards the ReduceScatter
// just wrote stay).
__device__ __forceinline__ void st16_stream(void* p, uint4 v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

// 16 bytes at an address aligned only to the element size ES (a shard whose
// start is not on a 16-byte boundary): the widest accesses the address
// allows, 16, 8, 4 or 2 bytes.  Little-endian: byte 0 is the low byte of x.
template <int ES>
__host__ __device__ __forceinline__ void st_aligned(void* p, const uint4& v) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if ((a & 15) == 0) {
        st16(p, v);
    } else if (ES >= 8 || (a & 7) == 0) {
        uint2* d = static_cast<uint2*>(p);
        d[0] = make_uint2(v.x, v.y);
        d[1] = make_uint2(v.z, v.w);
    } else if (ES >= 4 || (a & 3) == 0) {
        unsigned* d = static_cast<unsigned*>(p);
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
    } else {
        unsigned short* d = static_cast<unsigned short*>(p);
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            d[2 * k] = (unsigned short)(w[k] & 0xffffu);
            d[2 * k + 1] = (unsigned short)(w[k] >> 16);
        }
    }
}

template <int ES>
__host__ __device__ __forceinline__ uint4 ld_aligned(const void* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    uint4 v;
    if ((a & 15) == 0) {
        v = ld16(p);
    } else if (ES >= 8 || (a & 7) == 0) {
        const uint2* s = static_cast<const uint2*>(p);
        const uint2 lo = s[0], hi = s[1];
        v = make_uint4(lo.x, lo.y, hi.x, hi.y);
    } else if (ES >= 4 || (a & 3) == 0) {
        const unsigned* s = static_cast<const unsigned*>(p);
        v = make_uint4(s[0], s[1], s[2], s[3]);
    } else {
        const unsigned short* s = static_cast<const unsigned short*>(p);
        unsigned w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = (unsigned)s[2 * k] | ((unsigned)s[2 * k + 1] << 16);
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return v;
}

// ------------------------------------------------ warp-realigned access --
//
// A ReduceScatter writes, and an AllGather reads, a shard at offset i - cq of
// the index i; when q elements are not a whole number of 16-byte vectors,
// that offset is off the 16-byte grid by d bytes (the same d for the whole
// shard).  A warp whose 32 lanes hold 32 consecutive vectors of one shard
// (512 contiguous bytes) then realigns them among its lanes: lane t accesses
// the aligned 16-byte block that starts d bytes before its own vector, and
// takes the other part from its neighbour by shuffle.  Only the first lane
// (the part of its block that lies inside the warp's bytes) and the last (the
// d bytes past its block) access single elements; every byte accessed lies
// inside the warp's 512 bytes.  All 32 lanes must call these together.
//
// Used for 2-byte elements only, where an off-grid vector otherwise takes
// eight 2-byte accesses.  Measured on GB300 (64 MiB per rank, shards off the
// grid): bf16 ReduceScatter at 3 ranks 0.68x -> 0.83x of the copy rate,
// AllGather 0.91x -> 0.94x.  With 4- and 8-byte elements (at most four
// accesses per vector) and in the streaming folds (N > 8 or run-time N), the
// extra instructions cost as much as they save or more, so those keep the
// element-aligned accesses.

constexpr unsigned kFullWarp = 0xffffffffu;

// Bytes [4*A0 + sh/8, ... + 16) of the 32-byte sequence w[0..7].
template <int A0>
__device__ __forceinline__ uint4 window_at(const unsigned (&w)[8], unsigned sh) {
    return make_uint4(__funnelshift_r(w[A0], w[A0 + 1], sh), __funnelshift_r(w[A0 + 1], w[A0 + 2], sh),
                      __funnelshift_r(w[A0 + 2], w[A0 + 3], sh),
                      __funnelshift_r(w[A0 + 3], w[A0 + 4], sh));
}

// Bytes [off, off + 16) of the 32 bytes lo ++ hi, 0 < off < 16.
__device__ __forceinline__ uint4 byte_window(const uint4& lo, const uint4& hi, int off) {
    const unsigned w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const unsigned sh = (unsigned)(off & 3) * 8u;
    switch (off >> 2) {
    case 0: return window_at<0>(w, sh);
    case 1: return window_at<1>(w, sh);
    case 2: return window_at<2>(w, sh);
    default: return window_at<3>(w, sh);
    }
}

__device__ __forceinline__ uint4 shfl_up1(const uint4& v) {
    return make_uint4(__shfl_up_sync(kFullWarp, v.x, 1), __shfl_up_sync(kFullWarp, v.y, 1),
                      __shfl_up_sync(kFullWarp, v.z, 1), __shfl_up_sync(kFullWarp, v.w, 1));
}

__device__ __forceinline__ uint4 shfl_down1(const uint4& v) {
    return make_uint4(__shfl_down_sync(kFullWarp, v.x, 1), __shfl_down_sync(kFullWarp, v.y, 1),
                      __shfl_down_sync(kFullWarp, v.z, 1), __shfl_down_sync(kFullWarp, v.w, 1));
}

// Element k (of 16/ES) of v.  Called from fully unrolled loops, so k is a
// constant after unrolling and the word index folds away.
template <int ES>
__host__ __device__ __forceinline__ unsigned long long elem_get(const uint4& v, int k) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (ES == 2) return (w[k / 2] >> (16 * (k % 2))) & 0xffffu;
    else if constexpr (ES == 4) return w[k];
    else return ((unsigned long long)w[2 * k + 1] << 32) | w[2 * k];
}

// Stores bytes [from, from + len) of v at p (the destination of byte
// `from`), one element at a time; from and len are multiples of ES.
template <int ES>
__host__ __device__ __forceinline__ void st_bytes(unsigned char* p, const uint4& v, int from, int len) {
#pragma unroll
    for (int k = 0; k < 16 / ES; ++k) {
        const int b = k * ES;
        if (b >= from && b < from + len) {
            unsigned char* e = p + (b - from);
            if constexpr (ES == 2) {
                *reinterpret_cast<unsigned short*>(e) = (unsigned short)elem_get<ES>(v, k);
            } else if constexpr (ES == 4) {
                *reinterpret_cast<unsigned*>(e) = (unsigned)elem_get<ES>(v, k);
            } else {
                *reinterpret_cast<unsigned long long*>(e) = elem_get<ES>(v, k);
            }
        }
    }
}

// Loads bytes [from, to) of the aligned 16-byte block at blk into the same
// byte positions of the result (the other bytes are zero), one element at a
// time; from and to are multiples of ES.
template <int ES>
__host__ __device__ __forceinline__ uint4 ld_block_part(const unsigned char* blk, int from, int to) {
    unsigned w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 16 / ES; ++k) {
        const int b = k * ES;
        if (b >= from && b < to) {
            if constexpr (ES == 2) {
                w[k / 2] |= (unsigned)*reinterpret_cast<const unsigned short*>(blk + b) << (16 * (k % 2));
            } else if constexpr (ES == 4) {
                w[k] = *reinterpret_cast<const unsigned*>(blk + b);
            } else {
                const unsigned long long e = *reinterpret_cast<const unsigned long long*>(blk + b);
                w[2 * k] = (unsigned)e;
                w[2 * k + 1] = (unsigned)(e >> 32);
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Lane t stores v, the t-th of the warp's 32 consecutive vectors, at dst.
template <int ES>
__device__ __forceinline__ void st_warp_realigned(void* dst, const uint4& v) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    const int d = (int)(a & 15);
    if (d == 0) {
        st16(dst, v);
        return;
    }
    const int lane = (int)(threadIdx.x & 31);
    const uint4 prev = shfl_up1(v);
    unsigned char* blk = reinterpret_cast<unsigned char*>(a - (uintptr_t)d);
    // the aligned block holding this vector's first 16 - d bytes: its first
    // d bytes are the previous lane's last d (lane 0 stores only its own
    // first 16 - d bytes)
    if (lane > 0)
        st16(blk, byte_window(prev, v, 16 - d));
    else
        st_bytes<ES>(static_cast<unsigned char*>(dst), v, 0, 16 - d);
    // the last lane's final d bytes open the next block
    if (lane == 31) st_bytes<ES>(blk + 16, v, 16 - d, d);
}

// Lane t loads the t-th of the warp's 32 consecutive vectors, at src.
template <int ES>
__device__ __forceinline__ uint4 ld_warp_realigned(const void* src) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src);
    const int d = (int)(a & 15);
    if (d == 0) return ld16(src);
    const int lane = (int)(threadIdx.x & 31);
    const unsigned char* blk = reinterpret_cast<const unsigned char*>(a - (uintptr_t)d);
    // this lane's aligned block (lane 0: only its bytes d..15, the others
    // lie before the warp's range); the vector is its bytes d..15 followed by
    // the first d bytes of the next block
    const uint4 cur = lane > 0 ? ld16(blk) : ld_block_part<ES>(blk, d, 16);
    uint4 next = shfl_down1(cur);
    if (lane == 31) next = ld_block_part<ES>(blk + 16, 0, d);
    return byte_window(cur, next, d);
}

// ------------------------------------------------------------------- ops --

// Two float lanes in one 64-bit register (lane 0 in the low half), for the
// paired single-precision instructions: each lane is one IEEE single
// operation rounded to nearest even, as __fadd_rn / __fmul_rn give, in half
// the instructions.
__device__ __forceinline__ unsigned long long f32x2(float lo, float hi) {
    return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f32x2_lo(unsigned long long v) { return __uint_as_float((unsigned)v); }
__device__ __forceinline__ float f32x2_hi(unsigned long long v) {
    return __uint_as_float((unsigned)(v >> 32));
}

// a (+) b with the running value on the left.  Floats: one IEEE single
// operation, explicitly rounded (no contraction into FMA); SUM and PROD also
// have the paired form apply2.  Integers: wrap modulo 2^64.  MAX/MIN keep a
// on ties.
struct OpSum {
    static constexpr bool kPaired = true;
    __device__ static __forceinline__ float apply(float a, float b) { return __fadd_rn(a, b); }
    __device__ static __forceinline__ long long apply(long long a, long long b) {
        return (long long)((unsigned long long)a + (unsigned long long)b);
    }
    __device__ static __forceinline__ unsigned long long apply2(unsigned long long a,
                                                               unsigned long long b) {
        unsigned long long r;
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
        return r;
    }
};
struct OpProd {
    static constexpr bool kPaired = true;
    __device__ static __forceinline__ float apply(float a, float b) { return __fmul_rn(a, b); }
    __device__ static __forceinline__ long long apply(long long a, long long b) {
        return (long long)((unsigned long long)a * (unsigned long long)b);
    }
    __device__ static __forceinline__ unsigned long long apply2(unsigned long long a,
                                                               unsigned long long b) {
        unsigned long long r;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
        return r;
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

// Whether Op has the paired float form (sum and product; max and min do not).
template <class Op, class = void> struct HasPaired : std::false_type {};
template <class Op> struct HasPaired<Op, std::void_t<decltype(Op::kPaired)>> : std::true_type {};

// The paired form serves the eight fp32 lanes of a bf16 vector only.  For
// fp32's four lanes it measured no gain, and building the register pairs
// pushed the fp32 trees with a run-time N over 128 registers into spills
// (fp32 ReduceScatter, tree order, 12 ranks: 1.02x -> 0.68x of the copy
// peak).
template <class Op, class A, int W>
__device__ __forceinline__ Vec<A, W> vop(const Vec<A, W>& a, const Vec<A, W>& b) {
    Vec<A, W> r;
    if constexpr (std::is_same<A, float>::value && W == 8 && HasPaired<Op>::value) {
#pragma unroll
        for (int k = 0; k < W; k += 2) {
            const unsigned long long v =
                Op::apply2(f32x2(a.x[k], a.x[k + 1]), f32x2(b.x[k], b.x[k + 1]));
            r.x[k] = f32x2_lo(v);
            r.x[k + 1] = f32x2_hi(v);
        }
    } else {
#pragma unroll
        for (int k = 0; k < W; ++k) r.x[k] = Op::apply(a.x[k], b.x[k]);
    }
    return r;
}

// AVG: one division by n after the ordered sum, correctly rounded.  For n a
// power of two, 1/n = 2^-k is exact in binary, so s * 2^-k is the same real
// number as s / n, and the correctly rounded product has the bits of the
// correctly rounded quotient (subnormal results included; infinities stay
// infinite): one multiply instead of a division.  Measured on GB300, the
// bf16 ReduceScatter of a 25 MiB gradient bucket on eight ranks went from
// 0.89x to 0.92x of the copy rate with AVG.  Other n divide.
__device__ __forceinline__ float avg_div(float s, int n) {
    if ((n & (n - 1)) == 0) {
        const int k = __ffs(n) - 1;  // n = 2^k, 0 <= k <= 6
        return __fmul_rn(s, __int_as_float((127 - k) << 23));
    }
    return __fdiv_rn(s, (float)n);
}
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

// The rank that plays node k of the tree in the second tree of a double
// binary tree: k + 1 mod n for even n (rank numbers shifted by one), n-1-k
// for odd n (the mirror image).
__host__ __device__ constexpr int tree_b_rank(int k, int n) {
    return (n % 2 == 0) ? (k + 1 == n ? 0 : k + 1) : n - 1 - k;
}

// The second tree with N known at compile time: every rank index stays a
// compile-time constant.
template <class L, int N> struct TreeBStatic {
    using A = typename L::A;
    static constexpr int W = L::W;
    using Raw = typename L::Raw;
    const L& l;
    __device__ __forceinline__ Raw raw(int k) const { return l.raw(tree_b_rank(k, N)); }
    __device__ __forceinline__ Vec<A, W> cvt(const Raw& r) const { return l.cvt(r); }
};

// The second tree with a run-time N (the rank index is computed).
template <class L> struct TreeBRuntime {
    using A = typename L::A;
    static constexpr int W = L::W;
    using Raw = typename L::Raw;
    const L& l;
    int n;
    __device__ __forceinline__ Raw raw(int k) const { return l.raw(tree_b_rank(k, n)); }
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

// Ring with a run-time N, read from a doubled pointer table (entry k holds
// rank k mod N), so the ranks c, c+1, ..., c+N-1 of chunk c are the entries
// c .. c+N-1 and need no wrap-around.  Whole groups of kGroup entries, then
// one group of the remaining N mod kGroup; each group's loads are all issued
// before it is folded, and no load needs a guard.
template <class Op, int R, class L>
__device__ __forceinline__ void ring_run(const L& ld, int k, VecOf<L>& acc, bool first) {
    typename L::Raw t[R];
#pragma unroll
    for (int u = 0; u < R; ++u) t[u] = ld.raw(k + u);
    if (first)
        acc = ld.cvt(t[0]);
    else
        acc = vop<Op>(acc, ld.cvt(t[0]));
#pragma unroll
    for (int u = 1; u < R; ++u) acc = vop<Op>(acc, ld.cvt(t[u]));
}

template <class Op, int R, class L>
__device__ __forceinline__ void ring_tail(const L& ld, int k, int rem, VecOf<L>& acc, bool first) {
    if constexpr (R > 0) {
        if (rem == R)
            ring_run<Op, R>(ld, k, acc, first);
        else
            ring_tail<Op, R - 1>(ld, k, rem, acc, first);
    }
}

template <class Op, class L>
__device__ __forceinline__ VecOf<L> fold_ring_doubled(const L& ld, int n, int c) {
    VecOf<L> acc;
    const int end = c + n;
    int k = c;
    bool first = true;
#pragma unroll 1
    for (; k + kGroup <= end; k += kGroup) {
        ring_run<Op, kGroup>(ld, k, acc, first);
        first = false;
    }
    ring_tail<Op, kGroup - 1>(ld, k, end - k, acc, first);
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

// Trees over n ranks, n not a power of two: the tree of the next power of
// two PT with ranks n .. PT-1 missing.  A node whose own rank is missing has
// nothing in its right subtree either, and passes its left subtree's value
// through; a present node whose right subtree is empty combines its left
// subtree with its own operand.  This is the tree in which a rank whose
// parent label (r - L) | 2L is not a rank hangs under r - L.  Each function
// is called only for a subtree that holds at least one rank.  With n a
// compile-time constant every test folds away; with a run-time n they are
// uniform branches.

// t[K] holds rank BASE + K (absent ranks are never read).  A subtree whose
// ranks all exist (its last rank P + L - 1 below n) takes the unchecked
// evaluation: with a run-time n the checks otherwise cost every node of
// every vector a compare and a branch (bf16 ReduceScatter over 12 ranks in
// the tree order ran 26 % more instructions than the ring).
template <class Op, int K, int L, class Ld, class R, int G>
__device__ __forceinline__ VecOf<Ld> tree_local_n(const Ld& ld, const R (&t)[G], int base, int n) {
    if constexpr (L == 1) {
        return ld.cvt(t[K]);
    } else {
        const int P = base + K;
        if (P + L - 1 < n) return tree_local<Op, K, L>(ld, t);
        VecOf<Ld> l = tree_local_n<Op, K - L / 2, L / 2>(ld, t, base, n);
        if (P >= n) return l;
        if (P + 1 >= n) return vop<Op>(l, ld.cvt(t[K]));
        VecOf<Ld> r = tree_local_n<Op, K + L / 2, L / 2>(ld, t, base, n);
        return vop<Op>(vop<Op>(l, r), ld.cvt(t[K]));
    }
}

// Block B of 16 ranks, as in tree_block, with the ranks from n on skipped.
template <class Op, int B, class Ld>
__device__ __forceinline__ VecOf<Ld> tree_block_n(const Ld& ld, typename Ld::Raw& first, int n) {
    typename Ld::Raw t[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) t[k] = (16 * B + k < n) ? ld.raw(16 * B + k) : typename Ld::Raw{};
    first = t[0];
    return tree_local_n<Op, 8, 8>(ld, t, 16 * B, n);
}

// T(P) for a node of level L >= 8, as in tree_upper.
template <class Op, int P, int L, class Ld>
__device__ __forceinline__ VecOf<Ld> tree_upper_n(const Ld& ld, typename Ld::Raw& first, int n) {
    if constexpr (L == 8) {
        return tree_block_n<Op, (P - 8) / 16>(ld, first, n);
    } else {
        VecOf<Ld> l = tree_upper_n<Op, P - L / 2, L / 2>(ld, first, n);
        if (P >= n) return l;
        if (P + 1 >= n) return vop<Op>(l, ld.cvt(ld.raw(P)));
        typename Ld::Raw own;
        VecOf<Ld> r = tree_upper_n<Op, P + L / 2, L / 2>(ld, own, n);
        return vop<Op>(vop<Op>(l, r), ld.cvt(own));
    }
}

// The root, rank 0, with the single child PT/2 (n >= 2).
template <class Op, int PT, class Ld>
__device__ __forceinline__ VecOf<Ld> fold_tree_n(const Ld& ld, int n) {
    static_assert(PT >= 4 && (PT & (PT - 1)) == 0, "envelope must be a power of two >= 4");
    if constexpr (PT >= 16) {
        typename Ld::Raw own0;
        VecOf<Ld> t = tree_upper_n<Op, PT / 2, PT / 2>(ld, own0, n);
        return vop<Op>(t, ld.cvt(own0));
    } else {
        typename Ld::Raw t[PT];
#pragma unroll
        for (int k = 0; k < PT; ++k) t[k] = (k < n) ? ld.raw(k) : typename Ld::Raw{};
        return vop<Op>(tree_local_n<Op, PT / 2, PT / 2>(ld, t, 0, n), ld.cvt(t[0]));
    }
}

__host__ __device__ constexpr bool is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }
__host__ __device__ constexpr int pow2_ceil(int n) { return n <= 1 ? 1 : 2 * pow2_ceil((n + 1) / 2); }

// One tree over the loader's ranks: NT > 0 a compile-time N (a power of two
// takes the plain tree), NT < 0 a run-time n inside the envelope -NT.
template <class Op, int NT, class Ld>
__device__ __forceinline__ VecOf<Ld> fold_any_tree(const Ld& ld, int n) {
    if constexpr (NT < 0) {
        return fold_tree_n<Op, -NT>(ld, n);
    } else if constexpr (is_pow2(NT)) {
        return fold_tree<Op, NT>(ld);
    } else {
        return fold_tree_n<Op, (pow2_ceil(NT) < 4 ? 4 : pow2_ceil(NT))>(ld, NT);
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

// NT > 0: N is a compile-time constant; NT == 0: ring with a run-time N;
// NT < 0: tree orders with a run-time N inside the envelope -NT.  The ring
// switches among its rotations up to N = 8 and folds in groups with
// run-time rank indices beyond.  `sel` is the ring's chunk, or for the
// double binary tree which tree (0 = A, 1 = B) the element belongs to.
template <class Op, int ORDER, int NT, class L>
__device__ __forceinline__ VecOf<L> fold(const L& ld, int n, int sel) {
    const int c = sel;
    if constexpr (ORDER == kOrderRecursiveHalving) {
        return rh_group<Op, 0, 1, NT>(ld);
    } else if constexpr (ORDER == kOrderPairwiseTree) {
        return fold_any_tree<Op, NT>(ld, n);
    } else if constexpr (ORDER == kOrderDoubleTree) {
        if (sel == 0) return fold_any_tree<Op, NT>(ld, n);
        if constexpr (NT > 0) {
            TreeBStatic<L, NT> b{ld};
            return fold_any_tree<Op, NT>(b, NT);
        } else {
            TreeBRuntime<L> b{ld, n};
            return fold_any_tree<Op, NT>(b, n);
        }
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
// AllReduce, all N outputs; ReduceScatter, the shard that owns it (realigned
// across the warp when `warp_shard`: the whole warp stores 32 consecutive
// vectors of that shard together).
template <class T, int NT, bool RS, class A, int V>
__device__ __forceinline__ void store_result(const ReduceParams& p, int c, long long i0,
                                             Vec<A, V>& acc, bool warp_shard) {
    if (p.avg) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
    }
    if constexpr (RS) {
        T* dst = static_cast<T*>(p.out[c]) + (i0 - (long long)c * p.q);
        if (warp_shard)
            st_warp_realigned<sizeof(T)>(dst, pack(acc, (T*)nullptr));
        else
            st_aligned<sizeof(T)>(dst, pack(acc, (T*)nullptr));
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

// The lanes of a vector that straddles a chunk boundary (or the double
// tree's halfway point) whose selector is `sel`, stored element by element:
// lane k holds element i0 + k of chunk c (c + 1 from `cut` on).
template <class T, int ORDER, bool RS, class A, int V>
__device__ __forceinline__ void store_lanes(const ReduceParams& p, int c, long long cut,
                                            long long i0, const Vec<A, V>& acc, int sel) {
#pragma unroll
    for (int k = 0; k < V; ++k) {
        const long long i = i0 + k;
        const int ci = i >= cut ? c + 1 : c;
        const int si = (ORDER == kOrderRing) ? ci
                     : (ORDER == kOrderDoubleTree ? (int)(i >= p.half) : 0);
        if (si != sel) continue;
        A r = acc.x[k];
        if (p.avg) r = avg_div(r, p.n);
        if constexpr (RS) {
            store1(static_cast<T*>(p.out[ci]) + (i - (long long)ci * p.q), r);
        } else {
            for (int s = 0; s < p.nout; ++s) store1(static_cast<T*>(p.out[s]) + i, r);
        }
    }
}

// One vector slot on its own, in the kernels with a compile-time N: the
// vector path if it lies inside one chunk and inside the data on aligned
// bases; inside the data but across a chunk boundary or the double tree's
// halfway point, the N operand vectors load whole and the fold runs once
// per selector among the lanes (each lane keeps its own); else (misaligned
// bases, the end of the data, the padding, shards shorter than a vector)
// element by element.  Element by element, a straddling vector's thread
// waited for one round of loads per element and finished microseconds
// after the rest of the grid (fp32 ReduceScatter, 8 ranks x 1,000,003:
// 8.0 us per call against 6.1 us with M = 1,000,000).  The kernel calls this
// only from whole warps (see reduce_body).
template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __noinline__ void reduce_slot(const ReduceParams& p, long long v) {
    constexpr int V = Traits<T>::V;
    const long long i0 = v * V;
    const int c = chunk_of(i0, p.q, p.inv_q, p.n);
    const long long cut = (long long)(c + 1) * p.q;  // lanes from here are in chunk c + 1
    const bool one_chunk = i0 + V <= cut;
    if (p.vec_ok && i0 + V <= p.M && (one_chunk || p.q >= V)) {
        const int s0 = (ORDER == kOrderRing) ? c
                     : (ORDER == kOrderDoubleTree ? (int)(i0 >= p.half) : 0);
        const long long last = i0 + V - 1;
        const int s1 = (ORDER == kOrderRing) ? (one_chunk ? c : c + 1)
                     : (ORDER == kOrderDoubleTree ? (int)(last >= p.half) : 0);
        VecLoader<T> ld{p, i0};
        auto acc = fold<Op, ORDER, NT>(ld, p.n, s0);
        if (one_chunk && s0 == s1) {
            store_result<T, NT, RS>(p, c, i0, acc, false);
            return;
        }
        store_lanes<T, ORDER, RS>(p, c, cut, i0, acc, s0);
        if (s1 != s0) {
            acc = fold<Op, ORDER, NT>(ld, p.n, s1);
            store_lanes<T, ORDER, RS>(p, c, cut, i0, acc, s1);
        }
    } else {
        for (int k = 0; k < V && i0 + k < p.limit; ++k) reduce_one<T, Op, ORDER, NT, RS>(p, i0 + k);
    }
}

// One vector slot on its own, in the kernels with a run-time N (they stream
// their operands in groups, through the pointer table in shared memory).
// Inside the data on aligned bases, the N operand vectors load as whole
// vectors, in the vector path's groups, and every lane's element is folded
// at once, also when the vector straddles a chunk boundary (the ring folds
// the two parts from two different ranks, a ReduceScatter stores them to two
// shards) or the double binary tree's halfway point (two trees): the fold
// then runs once per selector among the lanes (at most two, since q >= V
// puts at most one chunk boundary in a vector, and there is one halfway
// point), and each run stores the lanes it serves, element by element.
// Element by element, each element's reduction waited for its own loads
// group after group, and the few threads on straddling vectors ran many
// microseconds after the rest of the grid (measured on GB300: bf16
// ReduceScatter over twelve ranks with shards off the 16-byte grid, one SM
// active 108 k cycles against 70 k on average, the call 47 % longer).  What
// remains element by element: misaligned bases, the end of the data, the
// padding, and shards shorter than a vector (tiny calls).
// Inlined into the kernel: called as a separate function from the lanes of
// a warp that leave the vector path while the others stay on it, it made
// those other lanes' results wrong on GB300 (a ReduceScatter over 33 ranks:
// every warp holding a straddling vector came out wrong; inlined, or called
// by whole warps, every element was right; caught by the parity tests).
// The kernels with a compile-time N keep the element path below: there
// each element issues its loads in groups of up to 16 at once, and inlining
// the vector path raised their registers (three blocks per SM down to two
// at N = 3 and 5; two down to one at N = 16, 32, 64).
template <class T, class Op, int ORDER, int NT, bool RS>
__device__ __forceinline__ void reduce_slot_streaming(const ReduceParams& p, const void* const* s_in,
                                                      long long v) {
    static_assert(NT <= 0, "the kernels with a run-time N only");
    constexpr int V = Traits<T>::V;
    using A = typename Traits<T>::Acc;
    const long long i0 = v * V;
    const int c = chunk_of(i0, p.q, p.inv_q, p.n);
    const long long cut = (long long)(c + 1) * p.q;  // lanes from here are in chunk c + 1
    const bool one_chunk = i0 + V <= cut;
    if (p.vec_ok && i0 + V <= p.M && (one_chunk || p.q >= V)) {
        // the fold's selector of element i in chunk ci: the ring's chunk,
        // the double tree's half; the other orders fold every element alike
        auto sel_of = [&](long long i, int ci) -> int {
            if constexpr (ORDER == kOrderRing) return ci;
            else if constexpr (ORDER == kOrderDoubleTree) return (int)(i >= p.half);
            else return 0;
        };
        const int s0 = sel_of(i0, c);
        const int s1 = sel_of(i0 + V - 1, one_chunk ? c : c + 1);
        const bool whole = one_chunk && s0 == s1;
        // the pointer table in shared memory, as the vector path reads it
        // (doubled for the ring, so its folds run in groups of 16 unwrapped)
        const SharedTableLoader<T> ld{s_in, i0};
#pragma unroll 1
        for (int pass = 0; pass < (s1 != s0 ? 2 : 1); ++pass) {
            const int sel = pass == 0 ? s0 : s1;
            Vec<A, V> acc;
            if constexpr (ORDER == kOrderRing)
                acc = fold_ring_doubled<Op>(ld, p.n, sel);
            else
                acc = fold<Op, ORDER, NT>(ld, p.n, sel);
            if (whole) {
                store_result<T, NT, RS>(p, c, i0, acc, false);
                continue;
            }
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const long long i = i0 + k;
                const int ci = i >= cut ? c + 1 : c;
                if (sel_of(i, ci) != sel) continue;
                A r = acc.x[k];
                if (p.avg) r = avg_div(r, p.n);
                if constexpr (RS) {
                    store1(static_cast<T*>(p.out[ci]) + (i - (long long)ci * p.q), r);
                } else {
                    for (int s = 0; s < p.nout; ++s) store1(static_cast<T*>(p.out[s]) + i, r);
                }
            }
        }
    } else {
        for (int k = 0; k < V && i0 + k < p.limit; ++k) reduce_one<T, Op, ORDER, NT, RS>(p, i0 + k);
    }
}

// The kernel body.  A block takes U*blockDim.x consecutive vectors per
// iteration; thread t owns the U vectors t, t + blockDim.x, ... of that
// range (each warp access is 512 contiguous bytes).  When all U vectors sit
// inside one chunk and inside the data on aligned bases (nearly always), the
// thread issues every load before it folds or stores anything:
//  - compile-time N <= 8 (0 < NT <= 8): the N x U vectors (at most 16) are
//    loaded into registers in rank order, with constant rank indices, then
//    folded slot by slot in the order's tree (the ring picks its rotation
//    by the chunk);
//  - otherwise (U = 1): the fold streams its operands in groups of kGroup.
//    The ring beyond 8 ranks reads its pointers from a shared-memory copy
//    of the table (doubled when N is a run-time value, so a rotation never
//    wraps), and so do the trees with a run-time N (tree B computes its
//    rank indices).
// Anything else goes slot by slot (reduce_slot, or reduce_slot_streaming
// with a run-time N).
template <class T, class Op, int ORDER, int NT, int U, bool RS>
__device__ __forceinline__ void reduce_body(const ReduceParams& p) {
    constexpr int V = Traits<T>::V;
    // Launched with programmatic stream serialization, this grid may be
    // scheduled while the kernel before it drains; wait for that kernel to
    // complete and its writes to be visible before touching global memory.
    // (After a kernel that never signals, or launched plainly, this returns
    // once that kernel has completed, or at once.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr bool kPre = (NT > 0 && NT <= 8);
    // ring beyond 8 ranks: rotated rank indices read from shared memory
    // (with a run-time N, a doubled input table: entry k is rank k mod N)
    constexpr bool kTable = (ORDER == kOrderRing && (NT == 0 || NT > 8));
    // trees with a run-time N: input pointers from shared memory (tree B
    // computes its rank indices)
    constexpr bool kTreeTable = (NT < 0);
    constexpr int kInEntries = (kTable && NT == 0) ? 2 * kMaxRanks
                                                    : ((kTable || kTreeTable) ? kMaxRanks : 1);
    __shared__ const void* s_in[kInEntries];
    __shared__ void* s_out[kTable ? kMaxRanks : 1];
    if constexpr (kTable || kTreeTable) {
        for (int r = threadIdx.x; r < p.n; r += blockDim.x) {
            s_in[r] = p.in[r];
            if constexpr (kTable && NT == 0) s_in[r + p.n] = p.in[r];
            if constexpr (kTable) s_out[r] = p.out[r];
        }
        __syncthreads();
    }
    const long long nvec = (p.limit + V - 1) / V;
    const long long span = (long long)blockDim.x * U;
    // With U > 1, the last span first, then the others in index order.  The
    // last span may hold only part of each thread's U vectors; those
    // threads reduce their vectors slot by slot, one round of loads after
    // another, and issued last, the span ended the kernel late.  Issued
    // first, its latency overlaps the rest of the grid.  Measured on GB300
    // (back-to-back calls, fraction of the copy peak): fp32 ReduceScatter
    // over 3 ranks x 64 MiB with M = 16,777,212, one vector short of a whole
    // number of spans, 0.93x -> 1.00x (1.01x at M = 16,777,216), the
    // AllReduce 0.94x -> 0.99x; 8 ranks x 1,000,003 0.72x -> 0.75x; whole
    // spans unchanged.  (The AllGather walks its spans from the end, so in
    // the decomposed AllReduce it still reads first the shards that this
    // kernel wrote last.)
    const long long last_b0 = (nvec - 1) / span * span;
    for (long long b = (long long)blockIdx.x * span; b < nvec; b += (long long)gridDim.x * span) {
        long long b0 = b;
        if constexpr (U > 1) b0 = (b == 0) ? last_b0 : b - span;
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
        // ReduceScatter of 2-byte elements with the operands preloaded: when
        // every lane of the warp takes the vector path into the same shard,
        // the warp's vectors of each slot are 512 contiguous bytes of that
        // shard, stored realigned (every lane of the
        // block reaches this point: the loop bounds are the same for all; the
        // shuffle runs in every lane, before the test: a lane that skipped it
        // would leave the others waiting in it)
        bool warp_shard = false;
        if constexpr (RS && kPre && sizeof(T) == 2) {
            const int c_lane0 = __shfl_sync(kFullWarp, c, 0);
            warp_shard = __all_sync(kFullWarp, wide && c == c_lane0);
        }
        // With a compile-time N, a warp with any lane off the vector path
        // sends every lane through reduce_slot, an out-of-line function, so
        // that it is never called from part of a warp while the rest of the
        // warp runs the vector path (a divergent call of that kind gave the
        // other lanes wrong results in the run-time-N kernels, which now
        // inline their slot path instead).  Every lane reaches this point.
        if constexpr (NT > 0) wide = __all_sync(kFullWarp, wide);
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
                    store_result<T, NT, RS>(p, c, (v0 + (long long)u * blockDim.x) * V, acc,
                                            warp_shard);
                }
            } else if constexpr (kTable) {
                static_assert(U == 1, "streaming folds take one vector per thread");
                SharedTableLoader<T> ld{s_in, v0 * V};
                VecOf<SharedTableLoader<T>> acc;
                if constexpr (NT == 0)
                    acc = fold_ring_doubled<Op>(ld, p.n, c);
                else
                    acc = fold<Op, ORDER, NT>(ld, p.n, c);
                if (p.avg) {
#pragma unroll
                    for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
                }
                const long long i0 = v0 * V;
                if constexpr (RS) {
                    T* dst = static_cast<T*>(s_out[c]) + (i0 - (long long)c * p.q);
                    st_aligned<sizeof(T)>(dst, pack(acc, (T*)nullptr));
                } else {
                    const uint4 u = pack(acc, (T*)nullptr);
                    for (int s = 0; s < p.nout; ++s) st16(static_cast<T*>(s_out[s]) + i0, u);
                }
            } else if constexpr (kTreeTable) {
                static_assert(U == 1, "streaming folds take one vector per thread");
                SharedTableLoader<T> ld{s_in, v0 * V};
                auto acc = fold<Op, ORDER, NT>(ld, p.n, sel);
                store_result<T, NT, RS>(p, c, v0 * V, acc, false);
            } else {
                static_assert(U == 1, "streaming folds take one vector per thread");
                VecLoader<T> ld{p, v0 * V};
                auto acc = fold<Op, ORDER, NT>(ld, p.n, sel);
                store_result<T, NT, RS>(p, c, v0 * V, acc, false);
            }
        } else {
#pragma unroll 1
            for (int u = 0; u < U; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) {
                    if constexpr (NT > 0)
                        reduce_slot<T, Op, ORDER, NT, RS>(p, v);
                    else
                        reduce_slot_streaming<T, Op, ORDER, NT, RS>(p, s_in, v);
                }
            }
        }
    }
    // This block is done: a kernel launched after this one with programmatic
    // stream serialization may start now (it waits for the whole grid, and
    // for its memory, before it touches any; see vc_ag_kernel).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Resident blocks per SM the reduction kernels ask ptxas for.  Compile-time
// N: one, stated explicitly.  Measured on GB300 against the bare launch
// bound: ptxas then keeps more loads in flight per thread, which lifts
// AllReduce by 0.5-1 % across the board and the 64-rank tree from 0.78x to
// 1.06x the copy rate (the one loss measured: bf16 RS at 32 ranks in the
// tree orders, 7.19 -> 6.54 TB/s).  Run-time N (folds that stream 16
// operands at a time): two, so that a second block hides the first one's
// load latency; measured, the ring at N = 12 went from 0.81x to 0.96x (bf16
// 0.67x to 0.82x).
//
// One exception: the bf16 ReduceScatter at N = 4 .. 8 asks for three blocks.
// At N = 4 and 8 its fold takes 87-88 registers under the one-block bound,
// just over the 85 that fit three blocks; bound to three it takes 76 with no
// spills.  The ReduceScatter, which reads N streams per store, gains from
// the extra warps' loads in flight: measured 0.5-1.5 points of the copy peak
// (N = 8 1.046x -> 1.052x, the 25 MiB bucket on 8 ranks 0.982x -> 0.993x);
// the AllReduce and the fp32 ReduceScatter gained nothing.  At N = 2 the
// same ReduceScatter asks for four (62 registers instead of 65-72, which
// left three): 2 x 64 MiB 0.97x -> 0.99x, with shards off the grid 0.90x
// -> 0.94x, 2 x 128 MiB 1.03x -> 1.02x; the fp32 kernel already runs four.
template <int NT, bool RS = false, int ES = 4>
constexpr int min_blocks() {
    if (NT <= 0) return 2;
    if (RS && ES == 2 && NT >= 4 && NT <= 8) return 3;
    if (RS && ES == 2 && NT == 2) return 4;
    return 1;
}

// ReduceScatter: index space [0, N*q), one store per element into the shard
// that owns it.
template <class T, class Op, int ORDER, int NT, int U>
__global__ void __launch_bounds__(kThreads, min_blocks<NT, true, sizeof(T)>()) vc_rs_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, U, true>(p);
}

// Fused AllReduce: index space [0, M), N stores per element (one, to the
// root's buffer, for Reduce).
template <class T, class Op, int ORDER, int NT, int U>
__global__ void __launch_bounds__(kThreads, min_blocks<NT>()) vc_ar_kernel(const __grid_constant__ ReduceParams p) {
    reduce_body<T, Op, ORDER, NT, U, false>(p);
}

// AllGather: output index i comes from shard s = floor(i/q) at offset i - sq,
// and is written to all N outputs.  It moves bits only, so it is typed by
// element size alone.  Like the reductions, a thread takes S
// vectors (blockDim.x apart) and loads all of them before it stores any.
// When the M output indices alone give too few blocks for the GPU (small M,
// many ranks), the outputs are split into groups along the grid's y axis:
// each group re-reads the (small) source and writes its share of the ranks.
template <int ES> struct Bits;
template <> struct Bits<2> { using U = unsigned short; };
template <> struct Bits<4> { using U = unsigned; };
template <> struct Bits<8> { using U = unsigned long long; };

// Vectors per thread: 8 when the call writes at least kGatherWideVectors
// 16-byte vectors in all (N outputs), 2 below.  Measured on GB300 (fp32):
// 2 gain 10-15 % at 2-64 MiB per rank (more, smaller blocks balance the last
// wave); 8 stay 1-4 % ahead once the outputs reach ~1 GiB (256 MiB x 4
// ranks, 32 MiB x 64 ranks).
constexpr long long kGatherWideVectors = 64LL << 20;  // 1 GiB of output

template <int ES>
__device__ __forceinline__ uint4 gather_load(const GatherParams& p, int s, long long i0) {
    using U = typename Bits<ES>::U;
    const U* src = static_cast<const U*>(p.in[s]) + (i0 - (long long)s * p.q);
    return ld_aligned<ES>(src);
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
        // every element's load first (they issue together), then the stores
        U val[V];
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const long long i = i0 + k;
            if (i < p.M) {
                const int si = chunk_of(i, p.q, p.inv_q, p.n);
                val[k] = static_cast<const U*>(p.in[si])[i - (long long)si * p.q];
            }
        }
#pragma unroll
        for (int k = 0; k < V; ++k)
            if (i0 + k < p.M)
                for (int r = r0; r < r1; ++r) static_cast<U*>(p.out[r])[i0 + k] = val[k];
    }
}

// REALIGN (2-byte elements only): some shard that the call reads sits off the
// 16-byte grid (q elements not a whole number of vectors, or a shard base off
// the grid); the host picks the instance, so every other call runs code
// without the warp-realigned loads.
template <int ES, int S, bool REALIGN>
__global__ void __launch_bounds__(kThreads) vc_ag_kernel(const __grid_constant__ GatherParams p) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
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
    // The spans are taken from the end of the index space: blocks start in
    // index order, so the first to run read the last shards, which a
    // ReduceScatter just before (the decomposed AllReduce) wrote last and
    // which are still in L2.  Taken from the start, they would be evicted by
    // this kernel's own writes before it reached them.
    const long long nspans = (nvec + span - 1) / span;
    for (long long j = blockIdx.x; j < nspans; j += gridDim.x) {
        const long long b0 = (nspans - 1 - j) * span;
        const long long v0 = b0 + threadIdx.x;
        const long long vlast = v0 + (long long)(S - 1) * blockDim.x;
        bool wide = false;
        int s = 0;
        if (vlast < nvec && p.vec_ok) {
            s = chunk_of(v0 * V, p.q, p.inv_q, p.n);
            const long long end = vlast * V + V;
            wide = end <= p.M && end <= (long long)(s + 1) * p.q;
        }
        // when every lane of the warp takes the vector path from the same
        // shard, the warp's vectors of each slot are 512 contiguous bytes of
        // it, loaded realigned (the loop bounds are the same for all lanes;
        // the shuffle runs in every lane, before the test: a lane that
        // skipped it would leave the others waiting in it)
        bool warp_shard = false;
        if constexpr (REALIGN) {
            const int s_lane0 = __shfl_sync(kFullWarp, s, 0);
            warp_shard = __all_sync(kFullWarp, wide && s == s_lane0);
        }
        if (wide) {
            uint4 val[S];
            if (warp_shard) {
                const U* src = static_cast<const U*>(p.in[s]) + (v0 * V - (long long)s * p.q);
#pragma unroll
                for (int u = 0; u < S; ++u)
                    val[u] = ld_warp_realigned<ES>(src + (long long)u * blockDim.x * V);
            } else {
#pragma unroll
                for (int u = 0; u < S; ++u)
                    val[u] = gather_load<ES>(p, s, (v0 + (long long)u * blockDim.x) * V);
            }
            // streaming stores from four outputs on (st16_stream); below
            // that they measured slower (3 ranks: bf16 with shards off the
            // grid 0.92x -> 0.88x of the copy peak, fp32 0.998x -> 0.992x)
            if (r1 - r0 >= 4) {
                for (int r = r0; r < r1; ++r) {
                    U* dst = static_cast<U*>(p.out[r]) + v0 * V;
#pragma unroll
                    for (int u = 0; u < S; ++u) st16_stream(dst + (long long)u * blockDim.x * V, val[u]);
                }
            } else {
                for (int r = r0; r < r1; ++r) {
                    U* dst = static_cast<U*>(p.out[r]) + v0 * V;
#pragma unroll
                    for (int u = 0; u < S; ++u) st16(dst + (long long)u * blockDim.x * V, val[u]);
                }
            }
        } else {
#pragma unroll 1
            for (int u = 0; u < S; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) gather_slot<ES>(p, v, r0, r1);
            }
        }
    }
    // this block is done: a kernel launched after this one may start
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches `kernel` with programmatic stream serialization: its grid may be
// scheduled while the kernel before it on the stream drains.  Every kernel
// launched this way executes griddepcontrol.wait before its first global
// access, so it still sees all of the preceding kernel's writes.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Launchers by element type (vc_reduce_dispatch.cu, which picks the slice of
// vc_reduce_inst.cu that holds the op and order).
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
