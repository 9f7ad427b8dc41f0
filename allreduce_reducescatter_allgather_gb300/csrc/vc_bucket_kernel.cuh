// The fused bucket kernels (see vc_bucket.cu for the host side): tiles of
// gradient tensors reduced where they are, in ring order with the ring chunk
// of their place in the bucket, and written either back to the N ranks'
// output tensors (AllReduce) or to the shard that owns the chunk
// (ReduceScatter).  (The AllGather of the shards back into the tensors moves
// bits only; its kernel is in vc_bucket.cu.)  Included by vc_bucket_inst.cu,
// which the build compiles once per element type.
#pragma once

#include <algorithm>

#include "vc.h"
#include "vc_device.cuh"

namespace vc {

struct BucketParams {
    const vc_bucket_tile_t* tiles;
    const void* const* in;   // reduction inputs, [tensor * n + rank]
    void* const* out;        // AllReduce / AllGather outputs, [tensor * n + rank]
    void* shard[kMaxRanks];  // shard r, q elements: ReduceScatter output, AllGather input
    long long q;             // ring chunk of the bucket: ceil(bucket_count / n)
    long long bucket_count;
    int ntiles;
    int n;
    int avg;
};

// One element of a rank's tensor, through the shared pointer table.
template <class T> struct SharedScalarLoader {
    using A = typename Traits<T>::Acc;
    static constexpr int W = 1;
    using Raw = A;
    const void* const* table;
    long long i;
    __device__ __forceinline__ Raw raw(int r) const {
        return load1(static_cast<const T*>(table[r]) + i);
    }
    __device__ __forceinline__ Vec<A, 1> cvt(const Raw& a) const {
        Vec<A, 1> v;
        v.x[0] = a;
        return v;
    }
};

// The reduced vector of tensor elements i0 .. i0+V-1 (bucket offset b0, in
// chunk c) to its destination: every rank's output tensor (AllReduce), or
// shard c at b0 - c*q (ReduceScatter; the shard's offset need not be on the
// 16-byte grid).
template <class T, bool RS, class Acc>
__device__ __forceinline__ void bucket_store(const BucketParams& p, void* const* s_out, int c,
                                             long long i0, long long b0, Acc& acc) {
    constexpr int V = Traits<T>::V;
    if (p.avg) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
    }
    const uint4 u = pack(acc, (T*)nullptr);
    if constexpr (RS) {
        st_aligned<sizeof(T)>(static_cast<T*>(p.shard[c]) + (b0 - (long long)c * p.q), u);
    } else {
        for (int r = 0; r < p.n; ++r) st16(static_cast<T*>(s_out[r]) + i0, u);
    }
}

template <class T, class Op, bool RS>
__device__ __forceinline__ void bucket_vector(const BucketParams& p, const void* const* s_in,
                                              void* const* s_out, int c, long long i0,
                                              long long b0) {
    SharedTableLoader<T> ld{s_in, i0};
    auto acc = fold_ring_doubled<Op>(ld, p.n, c);
    bucket_store<T, RS>(p, s_out, c, i0, b0, acc);
}

template <class T, class Op, bool RS>
__device__ __forceinline__ void bucket_element(const BucketParams& p, const void* const* s_in,
                                               void* const* s_out, int c, long long i,
                                               long long b) {
    using A = typename Traits<T>::Acc;
    SharedScalarLoader<T> ld{s_in, i};
    A val = fold_ring_doubled<Op>(ld, p.n, c).x[0];
    if (p.avg) val = avg_div(val, p.n);
    if constexpr (RS) {
        store1(static_cast<T*>(p.shard[c]) + (b - (long long)c * p.q), val);
    } else {
        for (int r = 0; r < p.n; ++r) store1(static_cast<T*>(s_out[r]) + i, val);
    }
}

// A tile as vc_bucket_plan makes it lies inside the bucket and inside one
// ring chunk.  Tiles planned for another bucket_count (or N) may not: their
// chunk index could name a shard or a ring rotation that does not exist.
// The kernels skip such a tile (every thread of the block sees the same
// tile, so the block stays uniform) instead of touching memory through it.
__device__ __forceinline__ bool tile_in_plan(const vc_bucket_tile_t& t, const BucketParams& p) {
    if (t.bucket_offset < 0 || t.count < 0 || t.bucket_offset + t.count > p.bucket_count)
        return false;
    const long long c = t.bucket_offset / p.q;
    return c < p.n && t.bucket_offset + t.count <= (c + 1) * p.q;
}

// ReduceScatter: the shard positions no tensor covers, from bucket offset
// lo to hi.  Below bucket_count they are the gaps between tensors, which
// the packed bucket holds as zeros on every rank: every op reduces zeros
// to zero.  From bucket_count on they are the padding up to N*q: the op's
// identity (0 for AVG), as the ReduceScatter pads.
template <class T, class Op>
__device__ __forceinline__ void bucket_fill(const BucketParams& p, long long lo, long long hi) {
    using A = typename Traits<T>::Acc;
    lo = lo < 0 ? 0 : lo;
    hi = hi > (long long)p.n * p.q ? (long long)p.n * p.q : hi;
    for (long long b = lo + threadIdx.x; b < hi; b += blockDim.x) {
        const int c = (int)(b / p.q);
        const A v = b < p.bucket_count ? A(0) : (p.avg ? A(0) : Identity<T, Op>::get());
        store1(static_cast<T*>(p.shard[c]) + (b - (long long)c * p.q), v);
    }
}

// NT > 0: N known at compile time; a thread loads the N x U operand vectors
// of its U vectors (blockDim.x apart) into registers before folding any, as
// the AllReduce kernel does; the slots of a span past the tile's last vector
// load and store nothing.  NT == 0: a run-time N, one vector at a time.
// The tiles come in bucket order (vc_bucket_plan writes them so); for the
// ReduceScatter, the block of tile t also fills the uncovered positions up
// to the next tile (tile 0's block, those before it too).
//
// Resident blocks: bf16 with N = 4 .. 8 asks for three (at most 80
// registers), everything else for two.  Measured on GB300 (a 24 MiB bucket
// of bf16 tensors on 8 ranks, ncu): at two blocks the ReduceScatter ran
// 19 % behind the ReduceScatter of the packed bucket, with the same DRAM
// bytes and two thirds of its warps.  The compile-time path then also
// handles a tile's partial last span itself (predicated loads) instead of
// the run-time-N vector fold, whose 16-operand groups set the kernel's
// register count (116 -> 76-80).  Each block sets up its tile (descriptor,
// then the N pointers into shared memory) before loading any operand; with
// three blocks per SM that latency overlaps the other blocks' streams, and
// prefetching the next tile's set-up measured no faster.  The bucket
// ReduceScatter of 351 MiB of bf16 tensors on 8 ranks: 559 -> 524 us (the
// packed bucket: 497 us); the AllReduce 921 -> 915 us (878 us).
template <class T, class Op, int NT, int U, bool RS>
__global__ void __launch_bounds__(kThreads, (sizeof(T) == 2 && NT >= 4 && NT <= 8) ? 3 : 2)
    vc_bucket_kernel(const __grid_constant__ BucketParams p) {
    constexpr int V = Traits<T>::V;
    __shared__ const void* s_in[2 * kMaxRanks];
    __shared__ void* s_out[RS ? 1 : kMaxRanks];
    // launched with programmatic stream serialization: wait for the kernel
    // before this one to complete (and its writes to be visible) first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int me = threadIdx.x;  // < kThreads; threads below n carry pointers
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const vc_bucket_tile_t tile = p.tiles[t];
        __syncthreads();  // the last tile's readers are done with the tables
        if (me < p.n) {
            const void* a = p.in[(long long)tile.tensor * p.n + me];
            s_in[me] = a;
            s_in[me + p.n] = a;
            if constexpr (!RS) s_out[me] = p.out[(long long)tile.tensor * p.n + me];
        }
        __syncthreads();
        const bool valid = tile_in_plan(tile, p);  // the same in every thread
        const int c = valid ? (int)(tile.bucket_offset / p.q) : 0;  // the tile's ring chunk
        const long long nvec = (valid && (tile.flags & 1)) ? tile.count / V : 0;
        const long long span = (long long)blockDim.x * U;
        for (long long b0 = 0; b0 < nvec; b0 += span) {
            const long long v0 = b0 + threadIdx.x;
            if constexpr (NT > 0) {
                uint4 buf[NT][U];
#pragma unroll
                for (int r = 0; r < NT; ++r) {
                    const T* base = static_cast<const T*>(s_in[r]) + tile.tensor_offset + v0 * V;
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        buf[r][u] = v0 + (long long)u * blockDim.x < nvec
                                        ? ld16(base + (long long)u * blockDim.x * V)
                                        : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (v0 + (long long)u * blockDim.x < nvec) {
                        PreLoader<T, NT, U> ld{buf, u};
                        auto acc = fold<Op, kOrderRing, NT>(ld, NT, c);
                        const long long j = (v0 + (long long)u * blockDim.x) * V;
                        bucket_store<T, RS>(p, s_out, c, tile.tensor_offset + j,
                                            tile.bucket_offset + j, acc);
                    }
                }
            } else {
#pragma unroll 1
                for (int u = 0; u < U; ++u) {
                    const long long v = v0 + (long long)u * blockDim.x;
                    if (v < nvec)
                        bucket_vector<T, Op, RS>(p, s_in, s_out, c, tile.tensor_offset + v * V,
                                                 tile.bucket_offset + v * V);
                }
            }
        }
        // the tile's tail, or all of it when its addresses are not aligned
        const long long tail_end = valid ? tile.count : 0;
        for (long long j = nvec * V + threadIdx.x; j < tail_end; j += blockDim.x)
            bucket_element<T, Op, RS>(p, s_in, s_out, c, tile.tensor_offset + j,
                                      tile.bucket_offset + j);
        if constexpr (RS) {
            if (valid) {
                const long long next_start =
                    t + 1 < p.ntiles ? p.tiles[t + 1].bucket_offset : (long long)p.n * p.q;
                if (t == 0) bucket_fill<T, Op>(p, 0, tile.bucket_offset);
                bucket_fill<T, Op>(p, tile.bucket_offset + tile.count, next_start);
            }
        }
    }
    // this block is done: a kernel launched after this one may start
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class T, class Op, int NT, int U>
cudaError_t launch_bucket_n(const BucketParams& p, bool rs, cudaStream_t st) {
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    // one block per tile up to 64 per SM, as the reduction kernels size
    // their grids (with 8 KiB tiles a 25 MiB bucket is ~3,200 tiles; capped
    // at 16 per SM, the bucket AllReduce of 351 MiB of bf16 tensors on 8
    // ranks measured 902 us against 897 us)
    const int blocks = std::min(p.ntiles, 64 * sms);
    if (rs) return launch_pdl(vc_bucket_kernel<T, Op, NT, U, true>, dim3(blocks), dim3(kThreads), st, p);
    return launch_pdl(vc_bucket_kernel<T, Op, NT, U, false>, dim3(blocks), dim3(kThreads), st, p);
}

// Compile-time N for the common rank counts (N x U at most 16 vectors of
// registers per thread), a run-time N otherwise.
template <class T, class Op>
cudaError_t launch_bucket_t(const BucketParams& p, bool rs, cudaStream_t st) {
    switch (p.n) {
    case 2: return launch_bucket_n<T, Op, 2, 4>(p, rs, st);
    case 4: return launch_bucket_n<T, Op, 4, 4>(p, rs, st);
    case 8: return launch_bucket_n<T, Op, 8, 2>(p, rs, st);
    default: return launch_bucket_n<T, Op, 0, 1>(p, rs, st);
    }
}

template <class T>
cudaError_t launch_bucket_op(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st) {
    switch (op) {
    case VC_SUM:
    case VC_AVG: return launch_bucket_t<T, OpSum>(p, rs, st);
    case VC_PROD: return launch_bucket_t<T, OpProd>(p, rs, st);
    case VC_MAX: return launch_bucket_t<T, OpMax>(p, rs, st);
    case VC_MIN: return launch_bucket_t<T, OpMin>(p, rs, st);
    default: return cudaErrorInvalidValue;
    }
}

// Launchers by element type (vc_bucket_inst.cu).
cudaError_t launch_bucket_i32(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st);
cudaError_t launch_bucket_i64(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st);
cudaError_t launch_bucket_f32(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st);
cudaError_t launch_bucket_bf16(const BucketParams& p, vc_op_t op, bool rs, cudaStream_t st);

}  // namespace vc
