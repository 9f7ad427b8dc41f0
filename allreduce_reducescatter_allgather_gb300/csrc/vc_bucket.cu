// vc_bucket_plan / vc_all_reduce_bucket / vc_reduce_scatter_bucket: the
// AllReduce or ReduceScatter of a gradient bucket whose tensors stay where
// they are.
//
// A DDP bucket ("通信与互联（01）" 三.1 and 九.1) is a flat buffer per rank
// into which many gradient tensors are packed, so one AllReduce replaces
// many small ones.  When the tensors live elsewhere, pack -> AllReduce ->
// unpack reads and writes every byte three times.  Here one kernel reads
// each tensor element from the N ranks' tensors, folds it in ring order with
// the ring chunk of its place in the bucket, and writes the result back to
// the N ranks' output tensors: the bits of the packed path, a third of its
// traffic, one launch.
//
// The host plan (vc_bucket_plan) lays the tensors out as the bucket would
// hold them and cuts them into tiles that never cross a ring chunk, so a
// tile's chunk is a constant.  The kernel takes tiles in a grid-stride loop;
// for each, the block copies the tensor's N input pointers (twice, so the
// ring's rotation never wraps) and N output pointers into shared memory.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "vc.h"
#include "vc_bucket_kernel.cuh"

namespace vc {
namespace {

// AllGather of the bucket: tile by tile, the shard of the tile's chunk
// (one read) into every rank's output tensor (N writes, with the
// AllGather's evict-first streaming stores: measured on GB300, the bucket
// AllGather of 351 MiB of bf16 tensors on 8 ranks 537 -> 526 us).  Moves
// bits only, so it is typed by element size.  A thread copies up to 2
// vectors per round, all loaded before any is stored.  Software-pipelined
// tile set-up: while a block works on tile t it has already fetched tile
// t + gridDim.x's descriptor and output pointers.  (Without it, and with
// the 48 registers that then allow five blocks per SM instead of four, the
// same AllGather measured 552 us.)
template <int ES>
__global__ void __launch_bounds__(kThreads) vc_bucket_gather_kernel(const __grid_constant__ BucketParams p) {
    using U = typename Bits<ES>::U;
    constexpr int V = 16 / ES;
    constexpr int S = 2;  // 256 threads x 2 vectors: a whole 8 KiB tile
    __shared__ void* s_out[kMaxRanks];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int t = blockIdx.x;
    if (t >= p.ntiles) return;
    vc_bucket_tile_t tile = p.tiles[t];
    const int me = threadIdx.x;
    void* my_out = me < p.n ? p.out[(long long)tile.tensor * p.n + me] : nullptr;
    for (; t < p.ntiles; t += gridDim.x) {
        __syncthreads();  // the last tile's writers are done with the table
        if (me < p.n) s_out[me] = my_out;
        __syncthreads();
        const int tn = t + gridDim.x;
        vc_bucket_tile_t next_tile = tile;
        if (tn < p.ntiles) next_tile = p.tiles[tn];
        // a tile planned for another bucket is skipped (tile_in_plan)
        const bool valid = tile_in_plan(tile, p);
        const int c = valid ? (int)(tile.bucket_offset / p.q) : 0;
        const U* src = static_cast<const U*>(p.shard[c]) + (valid ? tile.bucket_offset - (long long)c * p.q : 0);
        const long long nvec = (valid && (tile.flags & 1)) ? tile.count / V : 0;
        for (long long v0 = threadIdx.x; v0 < nvec; v0 += (long long)blockDim.x * S) {
            uint4 val[S];
#pragma unroll
            for (int u = 0; u < S; ++u) {
                const long long v = v0 + (long long)u * blockDim.x;
                if (v < nvec) val[u] = ld_aligned<ES>(src + v * V);
            }
            for (int r = 0; r < p.n; ++r) {
                U* dst = static_cast<U*>(s_out[r]) + tile.tensor_offset;
#pragma unroll
                for (int u = 0; u < S; ++u) {
                    const long long v = v0 + (long long)u * blockDim.x;
                    if (v < nvec) st16_stream(dst + v * V, val[u]);
                }
            }
        }
        const long long tail_end = valid ? tile.count : 0;
        for (long long j = nvec * V + threadIdx.x; j < tail_end; j += blockDim.x) {
            const U x = src[j];
            for (int r = 0; r < p.n; ++r) static_cast<U*>(s_out[r])[tile.tensor_offset + j] = x;
        }
        if (tn < p.ntiles) {
            tile = next_tile;
            if (me < p.n) my_out = p.out[(long long)tile.tensor * p.n + me];
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

int esize(vc_dtype_t dt) {
    switch (dt) {
    case VC_INT32: return 4;
    case VC_INT64: return 8;
    case VC_FLOAT32: return 4;
    case VC_BFLOAT16: return 2;
    default: return 0;
    }
}

bool launch_failure_injected() {
    const char* v = getenv("VC_TEST_FAIL_LAUNCH");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
}

struct Span {
    uintptr_t lo, hi;
    int tensor, rank;
};

// Outputs must not overlap each other; an input may overlap only its own
// output, exactly (in place).
vc_status_t check_bucket_alias(const std::vector<Span>& ins, std::vector<Span> outs) {
    std::sort(outs.begin(), outs.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    for (size_t k = 0; k + 1 < outs.size(); ++k)
        if (outs[k].hi > outs[k + 1].lo) return VC_ERR_ALIAS;
    for (const Span& s : ins) {
        // first output that ends after the input starts
        size_t lo = 0, hi = outs.size();
        while (lo < hi) {
            const size_t mid = (lo + hi) / 2;
            if (outs[mid].hi <= s.lo) lo = mid + 1; else hi = mid;
        }
        for (size_t k = lo; k < outs.size() && outs[k].lo < s.hi; ++k) {
            const Span& o = outs[k];
            const bool in_place = o.tensor == s.tensor && o.rank == s.rank && o.lo == s.lo &&
                                  o.hi == s.hi;
            if (!in_place) return VC_ERR_ALIAS;
        }
    }
    return VC_SUCCESS;
}

vc_status_t launch_bucket(const BucketParams& p, vc_dtype_t dtype, vc_op_t op, bool rs,
                          cudaStream_t st) {
    cudaError_t e;
    switch (dtype) {
    case VC_INT32: e = launch_bucket_i32(p, op, rs, st); break;
    case VC_INT64: e = launch_bucket_i64(p, op, rs, st); break;
    case VC_FLOAT32: e = launch_bucket_f32(p, op, rs, st); break;
    case VC_BFLOAT16: e = launch_bucket_bf16(p, op, rs, st); break;
    default: return VC_ERR_INVALID_ARGUMENT;
    }
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" vc_status_t vc_bucket_plan(const void* const* sendbufs, void* const* recvbufs,
                                      const size_t* counts, int ntensors, int nranks,
                                      vc_dtype_t dtype, vc_order_t order, vc_bucket_tile_t* tiles,
                                      int max_tiles, int* ntiles, size_t* bucket_count) {
    if (ntiles == nullptr || bucket_count == nullptr) return VC_ERR_INVALID_ARGUMENT;
    if (nranks < 1 || nranks > VC_MAX_RANKS || ntensors < 0 || max_tiles < 0)
        return VC_ERR_INVALID_ARGUMENT;
    const int es = esize(dtype);
    if (es == 0) return VC_ERR_INVALID_ARGUMENT;
    if (order < VC_ORDER_RING || order > VC_ORDER_DOUBLE_BINARY_TREE) return VC_ERR_INVALID_ARGUMENT;
    const bool is_float = dtype == VC_FLOAT32 || dtype == VC_BFLOAT16;
    if (order == VC_ORDER_RECURSIVE_HALVING && (nranks & (nranks - 1)) != 0)
        return VC_ERR_UNSUPPORTED;
    // floats: only the ring has a fused kernel; integers are order-free
    if (is_float && order != VC_ORDER_RING) return VC_ERR_UNSUPPORTED;
    if (ntensors > 0 && (sendbufs == nullptr || recvbufs == nullptr || counts == nullptr))
        return VC_ERR_INVALID_ARGUMENT;

    // the bucket layout: every tensor on a 16-byte boundary
    const unsigned long long align = 16 / es;
    const unsigned long long limit = (1ULL << 62) / (unsigned long long)es;
    std::vector<unsigned long long> base(ntensors);
    unsigned long long off = 0;
    std::vector<Span> ins, outs;
    for (int k = 0; k < ntensors; ++k) {
        base[k] = off;
        const unsigned long long c = counts[k];
        if (c > limit || off + c > limit) return VC_ERR_INVALID_ARGUMENT;
        off = (off + c + align - 1) / align * align;
        if (c == 0) continue;
        const size_t bytes = (size_t)c * es;
        for (int r = 0; r < nranks; ++r) {
            const void* in = sendbufs[(size_t)k * nranks + r];
            const void* out = recvbufs[(size_t)k * nranks + r];
            if (in == nullptr || out == nullptr) return VC_ERR_INVALID_ARGUMENT;
            if (reinterpret_cast<uintptr_t>(in) % es || reinterpret_cast<uintptr_t>(out) % es)
                return VC_ERR_INVALID_ARGUMENT;
            const uintptr_t i0 = reinterpret_cast<uintptr_t>(in);
            const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
            ins.push_back({i0, i0 + bytes, k, r});
            outs.push_back({o0, o0 + bytes, k, r});
        }
    }
    const vc_status_t a = check_bucket_alias(ins, outs);
    if (a != VC_SUCCESS) return a;

    // tiles: at most VC_BUCKET_TILE_MAX_BYTES, never across a ring chunk; a
    // tile that starts off the vector grid ends where the grid resumes, so
    // the tiles after it are aligned again (when the tensor's bases are)
    const unsigned long long total = off;
    const unsigned long long q = total == 0 ? 1 : (total + nranks - 1) / nranks;
    const unsigned long long tile_max = VC_BUCKET_TILE_MAX_BYTES / es;
    std::vector<vc_bucket_tile_t> plan;
    for (int k = 0; k < ntensors; ++k) {
        const unsigned long long c = counts[k];
        unsigned long long pos = 0;
        while (pos < c) {
            const unsigned long long b = base[k] + pos;
            const unsigned long long chunk_end = (b / q + 1) * q;
            unsigned long long len = std::min(c - pos, std::min(tile_max, chunk_end - b));
            if (pos % align != 0) len = std::min(len, align - pos % align);
            bool vec = true;
            for (int r = 0; r < nranks && vec; ++r) {
                const uintptr_t i = reinterpret_cast<uintptr_t>(sendbufs[(size_t)k * nranks + r]);
                const uintptr_t o = reinterpret_cast<uintptr_t>(recvbufs[(size_t)k * nranks + r]);
                vec = ((i + pos * es) % 16 == 0) && ((o + pos * es) % 16 == 0);
            }
            plan.push_back({(long long)b, (long long)pos, (long long)len, k, vec ? 1 : 0});
            pos += len;
        }
    }
    if (plan.size() > (size_t)0x7fffffff) return VC_ERR_INVALID_ARGUMENT;
    *ntiles = (int)plan.size();
    *bucket_count = (size_t)total;
    if (tiles == nullptr) return VC_SUCCESS;
    if (max_tiles < *ntiles) return VC_ERR_INVALID_ARGUMENT;
    if (!plan.empty()) std::memcpy(tiles, plan.data(), plan.size() * sizeof(vc_bucket_tile_t));
    return VC_SUCCESS;
}

extern "C" vc_status_t vc_all_reduce_bucket(const vc_bucket_tile_t* dev_tiles, int ntiles,
                                            const void* const* dev_sendbufs,
                                            void* const* dev_recvbufs, int nranks,
                                            size_t bucket_count, vc_dtype_t dtype, vc_op_t op,
                                            vc_stream_t stream) {
    if (nranks < 1 || nranks > VC_MAX_RANKS || ntiles < 0) return VC_ERR_INVALID_ARGUMENT;
    if (esize(dtype) == 0 || op < VC_SUM || op > VC_AVG) return VC_ERR_INVALID_ARGUMENT;
    if (ntiles == 0) return VC_SUCCESS;
    if (dev_tiles == nullptr || dev_sendbufs == nullptr || dev_recvbufs == nullptr ||
        bucket_count == 0)
        return VC_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(dev_tiles) % 8 != 0) return VC_ERR_INVALID_ARGUMENT;
    if (launch_failure_injected()) return VC_ERR_CUDA;
    BucketParams p = {};
    p.tiles = dev_tiles;
    p.in = dev_sendbufs;
    p.out = dev_recvbufs;
    p.q = (long long)((bucket_count + nranks - 1) / nranks);
    p.bucket_count = (long long)bucket_count;
    p.ntiles = ntiles;
    p.n = nranks;
    p.avg = op == VC_AVG;
    return launch_bucket(p, dtype, op, false, static_cast<cudaStream_t>(stream));
}

extern "C" vc_status_t vc_reduce_scatter_bucket(const vc_bucket_tile_t* dev_tiles, int ntiles,
                                                const void* const* dev_sendbufs,
                                                void* const* recvbufs, int nranks,
                                                size_t bucket_count, vc_dtype_t dtype,
                                                vc_op_t op, vc_stream_t stream) {
    if (nranks < 1 || nranks > VC_MAX_RANKS || ntiles < 0) return VC_ERR_INVALID_ARGUMENT;
    const int es = esize(dtype);
    if (es == 0 || op < VC_SUM || op > VC_AVG) return VC_ERR_INVALID_ARGUMENT;
    if (ntiles == 0) return VC_SUCCESS;
    if (dev_tiles == nullptr || dev_sendbufs == nullptr || recvbufs == nullptr ||
        bucket_count == 0)
        return VC_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(dev_tiles) % 8 != 0) return VC_ERR_INVALID_ARGUMENT;
    const unsigned long long q = (bucket_count + nranks - 1) / nranks;
    if (q > (1ULL << 62) / (unsigned long long)es) return VC_ERR_INVALID_ARGUMENT;
    std::vector<Span> shards;
    for (int r = 0; r < nranks; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(recvbufs[r]);
        if (a == 0 || a % es != 0) return VC_ERR_INVALID_ARGUMENT;
        shards.push_back({a, a + (uintptr_t)(q * es), -1, r});
    }
    const vc_status_t s = check_bucket_alias({}, shards);
    if (s != VC_SUCCESS) return s;
    if (launch_failure_injected()) return VC_ERR_CUDA;
    BucketParams p = {};
    p.tiles = dev_tiles;
    p.in = dev_sendbufs;
    p.out = nullptr;
    for (int r = 0; r < nranks; ++r) p.shard[r] = recvbufs[r];
    p.q = (long long)q;
    p.bucket_count = (long long)bucket_count;
    p.ntiles = ntiles;
    p.n = nranks;
    p.avg = op == VC_AVG;
    return launch_bucket(p, dtype, op, true, static_cast<cudaStream_t>(stream));
}

extern "C" vc_status_t vc_all_gather_bucket(const vc_bucket_tile_t* dev_tiles, int ntiles,
                                            const void* const* sendbufs, void* const* dev_recvbufs,
                                            int nranks, size_t bucket_count, vc_dtype_t dtype,
                                            vc_stream_t stream) {
    if (nranks < 1 || nranks > VC_MAX_RANKS || ntiles < 0) return VC_ERR_INVALID_ARGUMENT;
    const int es = esize(dtype);
    if (es == 0) return VC_ERR_INVALID_ARGUMENT;
    if (ntiles == 0) return VC_SUCCESS;
    if (dev_tiles == nullptr || sendbufs == nullptr || dev_recvbufs == nullptr ||
        bucket_count == 0)
        return VC_ERR_INVALID_ARGUMENT;
    if (reinterpret_cast<uintptr_t>(dev_tiles) % 8 != 0) return VC_ERR_INVALID_ARGUMENT;
    const unsigned long long q = (bucket_count + nranks - 1) / nranks;
    if (q > (1ULL << 62) / (unsigned long long)es) return VC_ERR_INVALID_ARGUMENT;
    for (int r = 0; r < nranks; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(sendbufs[r]);
        if (a == 0 || a % es != 0) return VC_ERR_INVALID_ARGUMENT;
    }
    if (launch_failure_injected()) return VC_ERR_CUDA;
    BucketParams p = {};
    p.tiles = dev_tiles;
    p.in = nullptr;
    p.out = dev_recvbufs;
    for (int r = 0; r < nranks; ++r) p.shard[r] = const_cast<void*>(sendbufs[r]);
    p.q = (long long)q;
    p.bucket_count = (long long)bucket_count;
    p.ntiles = ntiles;
    p.n = nranks;
    const int sms = sm_count();
    if (sms < 1) return VC_ERR_CUDA;
    const dim3 grid(std::min(ntiles, 16 * sms));
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (es) {
    case 2: e = launch_pdl(vc_bucket_gather_kernel<2>, grid, dim3(kThreads), st, p); break;
    case 4: e = launch_pdl(vc_bucket_gather_kernel<4>, grid, dim3(kThreads), st, p); break;
    default: e = launch_pdl(vc_bucket_gather_kernel<8>, grid, dim3(kThreads), st, p); break;
    }
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}
