// The fused bucket AllReduce kernel (see vc_bucket.cu for the host side):
// tiles of gradient tensors reduced where they are, in ring order with the
// ring chunk of their place in the bucket.  Included by vc_bucket_inst.cu,
// which the build compiles once per element type.
#pragma once

#include <algorithm>

#include "vc.h"
#include "vc_device.cuh"

namespace vc {

struct BucketParams {
    const vc_bucket_tile_t* tiles;
    const void* const* in;  // [tensor * n + rank]
    void* const* out;
    long long q;  // ring chunk of the bucket: ceil(bucket_count / n)
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

// One vector of consecutive tensor elements at tensor offset i0, reduced
// over the N ranks in ring order for chunk c and written to the N outputs.
template <class T, class Op>
__device__ __forceinline__ void bucket_vector(const BucketParams& p, const void* const* s_in,
                                              void* const* s_out, int c, long long i0) {
    constexpr int V = Traits<T>::V;
    SharedTableLoader<T> ld{s_in, i0};
    auto acc = fold_ring_doubled<Op>(ld, p.n, c);
    if (p.avg) {
#pragma unroll
        for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
    }
    const uint4 u = pack(acc, (T*)nullptr);
    for (int r = 0; r < p.n; ++r) st16(static_cast<T*>(s_out[r]) + i0, u);
}

// NT > 0: N known at compile time; a thread loads the N x U operand vectors
// of its U vectors (blockDim.x apart) into registers before folding any, as
// the AllReduce kernel does.  NT == 0: a run-time N, one vector at a time.
template <class T, class Op, int NT, int U>
__global__ void __launch_bounds__(kThreads, NT > 0 ? 1 : 2)
    vc_bucket_ar_kernel(const __grid_constant__ BucketParams p) {
    using A = typename Traits<T>::Acc;
    constexpr int V = Traits<T>::V;
    __shared__ const void* s_in[2 * kMaxRanks];
    __shared__ void* s_out[kMaxRanks];
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
        const vc_bucket_tile_t tile = p.tiles[t];
        __syncthreads();  // the last tile's readers are done with the tables
        for (int r = threadIdx.x; r < p.n; r += blockDim.x) {
            const void* a = p.in[(long long)tile.tensor * p.n + r];
            s_in[r] = a;
            s_in[r + p.n] = a;
            s_out[r] = p.out[(long long)tile.tensor * p.n + r];
        }
        __syncthreads();
        const int c = (int)(tile.bucket_offset / p.q);  // the tile's ring chunk
        const long long nvec = (tile.flags & 1) ? tile.count / V : 0;
        const long long span = (long long)blockDim.x * U;
        for (long long b0 = 0; b0 < nvec; b0 += span) {
            const long long v0 = b0 + threadIdx.x;
            if constexpr (NT > 0) {
                if (v0 + (long long)(U - 1) * blockDim.x < nvec) {
                    uint4 buf[NT][U];
#pragma unroll
                    for (int r = 0; r < NT; ++r) {
                        const T* base = static_cast<const T*>(s_in[r]) + tile.tensor_offset + v0 * V;
#pragma unroll
                        for (int u = 0; u < U; ++u) buf[r][u] = ld16(base + (long long)u * blockDim.x * V);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        PreLoader<T, NT, U> ld{buf, u};
                        auto acc = fold<Op, kOrderRing, NT>(ld, NT, c);
                        if (p.avg) {
#pragma unroll
                            for (int k = 0; k < V; ++k) acc.x[k] = avg_div(acc.x[k], p.n);
                        }
                        const uint4 w = pack(acc, (T*)nullptr);
                        const long long i0 = tile.tensor_offset + (v0 + (long long)u * blockDim.x) * V;
#pragma unroll
                        for (int r = 0; r < NT; ++r) st16(static_cast<T*>(s_out[r]) + i0, w);
                    }
                    continue;
                }
            }
#pragma unroll 1
            for (int u = 0; u < U; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) bucket_vector<T, Op>(p, s_in, s_out, c, tile.tensor_offset + v * V);
            }
        }
        // the tile's tail, or all of it when its addresses are not aligned
        for (long long j = nvec * V + threadIdx.x; j < tile.count; j += blockDim.x) {
            const long long i = tile.tensor_offset + j;
            SharedScalarLoader<T> ld{s_in, i};
            A val = fold_ring_doubled<Op>(ld, p.n, c).x[0];
            if (p.avg) val = avg_div(val, p.n);
            for (int r = 0; r < p.n; ++r) store1(static_cast<T*>(s_out[r]) + i, val);
        }
    }
}

template <class T, class Op, int NT, int U>
cudaError_t launch_bucket_n(const BucketParams& p, cudaStream_t st) {
    const int sms = sm_count();
    if (sms < 1) return cudaErrorInvalidDevice;
    const int blocks = std::min(p.ntiles, 16 * sms);
    vc_bucket_ar_kernel<T, Op, NT, U><<<blocks, kThreads, 0, st>>>(p);
    return cudaGetLastError();
}

// Compile-time N for the common rank counts (N x U at most 16 vectors of
// registers per thread), a run-time N otherwise.
template <class T, class Op>
cudaError_t launch_bucket_t(const BucketParams& p, cudaStream_t st) {
    switch (p.n) {
    case 2: return launch_bucket_n<T, Op, 2, 4>(p, st);
    case 4: return launch_bucket_n<T, Op, 4, 4>(p, st);
    case 8: return launch_bucket_n<T, Op, 8, 2>(p, st);
    default: return launch_bucket_n<T, Op, 0, 1>(p, st);
    }
}

template <class T>
cudaError_t launch_bucket_op(const BucketParams& p, vc_op_t op, cudaStream_t st) {
    switch (op) {
    case VC_SUM:
    case VC_AVG: return launch_bucket_t<T, OpSum>(p, st);
    case VC_PROD: return launch_bucket_t<T, OpProd>(p, st);
    case VC_MAX: return launch_bucket_t<T, OpMax>(p, st);
    case VC_MIN: return launch_bucket_t<T, OpMin>(p, st);
    default: return cudaErrorInvalidValue;
    }
}

// Launchers by element type (vc_bucket_inst.cu).
cudaError_t launch_bucket_i32(const BucketParams& p, vc_op_t op, cudaStream_t st);
cudaError_t launch_bucket_i64(const BucketParams& p, vc_op_t op, cudaStream_t st);
cudaError_t launch_bucket_f32(const BucketParams& p, vc_op_t op, cudaStream_t st);
cudaError_t launch_bucket_bf16(const BucketParams& p, vc_op_t op, cudaStream_t st);

}  // namespace vc
