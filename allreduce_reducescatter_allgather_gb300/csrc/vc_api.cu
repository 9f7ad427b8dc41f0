// The C ABI of include/vc.h: argument checks on the host, then one launch
// (two for the decomposed AllReduce) on the caller's stream.  Nothing is
// allocated; the pointer tables travel by value in the kernel parameters.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "vc.h"
#include "vc_device.cuh"

namespace vc {

namespace {

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlap(const Range& a, const Range& b) {
    return a.lo < b.hi && b.lo < a.hi && a.lo < a.hi && b.lo < b.hi;
}

int elem_size(vc_dtype_t dt) {
    switch (dt) {
    case VC_INT32: return 4;
    case VC_INT64: return 8;
    case VC_FLOAT32: return 4;
    case VC_BFLOAT16: return 2;
    default: return 0;
    }
}

bool valid_op(vc_op_t op) { return op >= VC_SUM && op <= VC_AVG; }
bool valid_order(vc_order_t o) {
    return o >= VC_ORDER_RING && o <= VC_ORDER_DOUBLE_BINARY_TREE;
}

// Common checks of every call.  *bytes_m and *bytes_q receive the byte sizes
// of a full rank buffer (M elements) and of a shard (q elements).
vc_status_t check_shape(int nranks, size_t count, vc_dtype_t dtype, size_t* bytes_m,
                        size_t* bytes_q) {
    if (nranks < 1 || nranks > VC_MAX_RANKS) return VC_ERR_INVALID_ARGUMENT;
    const int es = elem_size(dtype);
    if (es == 0) return VC_ERR_INVALID_ARGUMENT;
    // element indices are signed 64-bit in the kernels; byte sizes must fit
    if (count > (size_t)(1ULL << 62) / (size_t)es) return VC_ERR_INVALID_ARGUMENT;
    const size_t q = vc_shard_count(count, nranks);
    *bytes_m = count * (size_t)es;
    *bytes_q = q * (size_t)es;
    return VC_SUCCESS;
}

// Every buffer must be non-NULL and aligned to its element size (the
// kernels' element-wise paths access whole elements).
vc_status_t check_table(const void* const* t, int n, vc_dtype_t dtype) {
    if (t == nullptr) return VC_ERR_INVALID_ARGUMENT;
    const uintptr_t es = (uintptr_t)elem_size(dtype);
    for (int r = 0; r < n; ++r)
        if (t[r] == nullptr || reinterpret_cast<uintptr_t>(t[r]) % es != 0)
            return VC_ERR_INVALID_ARGUMENT;
    return VC_SUCCESS;
}

Range range_of(const void* p, size_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + bytes};
}

// Outputs must be pairwise disjoint and disjoint from every input, except
// that output r may be exactly input r when allow_in_place is set.
// O(N log N): the outputs are sorted by start address, so they are disjoint
// iff each ends before the next starts; an input can then only overlap the
// first output that ends after the input starts (outputs beyond it start
// later still), or -- when that one is its own in-place output, which ends
// exactly where the input ends -- none.
vc_status_t check_alias(const void* const* in, size_t in_bytes, void* const* out,
                        size_t out_bytes, int n, bool allow_in_place) {
    if (out_bytes == 0) return VC_SUCCESS;
    int order[VC_MAX_RANKS];
    for (int r = 0; r < n; ++r) order[r] = r;
    std::sort(order, order + n, [&](int a, int b) {
        return reinterpret_cast<uintptr_t>(out[a]) < reinterpret_cast<uintptr_t>(out[b]);
    });
    Range sorted[VC_MAX_RANKS];
    for (int k = 0; k < n; ++k) sorted[k] = range_of(out[order[k]], out_bytes);
    for (int k = 0; k + 1 < n; ++k)
        if (sorted[k].hi > sorted[k + 1].lo) return VC_ERR_ALIAS;
    if (in_bytes == 0) return VC_SUCCESS;
    for (int s = 0; s < n; ++s) {
        const Range i = range_of(in[s], in_bytes);
        // first output whose end lies beyond the input's start
        int lo = 0, hi = n;
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if (sorted[mid].hi <= i.lo) lo = mid + 1; else hi = mid;
        }
        if (lo == n || !overlap(sorted[lo], i)) continue;
        const int r = order[lo];
        const bool same = allow_in_place && r == s && in[s] == out[r] && in_bytes == out_bytes;
        if (!same) return VC_ERR_ALIAS;
    }
    return VC_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Test hook: with VC_TEST_FAIL_LAUNCH set to a non-zero value the next
// launches report a launch failure instead of launching.  Lets the error path
// be exercised without a faulty kernel.
bool injected_launch_failure() {
    const char* v = getenv("VC_TEST_FAIL_LAUNCH");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
}

// nout: outputs the AllReduce kernel writes (n, or 1 for Reduce); the
// ReduceScatter kernel always has n.
vc_status_t launch_reduce(const void* const* in, void* const* out, int n, size_t count,
                          vc_dtype_t dtype, vc_op_t op, vc_order_t order, bool rs,
                          cudaStream_t st, int nout = -1) {
    ReduceParams p;
    memset(&p, 0, sizeof p);
    const long long M = (long long)count;
    const long long q = (long long)vc_shard_count(count, n);
    if (nout < 0) nout = n;
    bool vec = true;
    for (int r = 0; r < n; ++r) {
        p.in[r] = in[r];
        vec = vec && aligned16(in[r]);
    }
    for (int r = 0; r < (rs ? n : nout); ++r) {
        p.out[r] = out[r];
        vec = vec && (rs || aligned16(out[r]));
    }
    p.nout = nout;
    p.M = M;
    p.q = q;
    p.limit = rs ? (long long)n * q : M;
    p.half = (M + 1) / 2;
    p.inv_q = 1.0f / (float)q;
    p.n = n;
    p.avg = (op == VC_AVG);
    p.vec_ok = vec;
    if (injected_launch_failure()) return VC_ERR_CUDA;
    cudaError_t e;
    switch (dtype) {
    case VC_INT32: e = launch_reduce_i32(p, (int)op, (int)order, rs, st); break;
    case VC_INT64: e = launch_reduce_i64(p, (int)op, (int)order, rs, st); break;
    case VC_FLOAT32: e = launch_reduce_f32(p, (int)op, (int)order, rs, st); break;
    case VC_BFLOAT16: e = launch_reduce_bf16(p, (int)op, (int)order, rs, st); break;
    default: return VC_ERR_INVALID_ARGUMENT;
    }
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}

vc_status_t launch_all_gather(const void* const* in, void* const* out, int n, size_t count,
                              vc_dtype_t dtype, cudaStream_t st) {
    GatherParams p;
    memset(&p, 0, sizeof p);
    bool vec = true;
    for (int r = 0; r < n; ++r) {
        p.in[r] = in[r];
        p.out[r] = out[r];
        vec = vec && aligned16(out[r]);
    }
    p.M = (long long)count;
    p.q = (long long)vc_shard_count(count, n);
    p.inv_q = 1.0f / (float)p.q;
    p.n = n;
    p.vec_ok = vec;
    if (injected_launch_failure()) return VC_ERR_CUDA;
    const cudaError_t e = launch_gather(p, elem_size(dtype), st);
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}

// Broadcast: every output receives the source buffer; the AllGather kernel
// with a single shard of q = M elements.
vc_status_t launch_broadcast(const void* src, void* const* out, int nout, size_t count,
                             vc_dtype_t dtype, cudaStream_t st) {
    if (nout == 0) return VC_SUCCESS;
    GatherParams p;
    memset(&p, 0, sizeof p);
    bool vec = true;
    p.in[0] = src;
    for (int r = 0; r < nout; ++r) {
        p.out[r] = out[r];
        vec = vec && aligned16(out[r]);
    }
    p.M = (long long)count;
    p.q = (long long)count;
    p.inv_q = 1.0f / (float)p.q;
    p.n = nout;
    p.vec_ok = vec;
    if (injected_launch_failure()) return VC_ERR_CUDA;
    const cudaError_t e = launch_gather(p, elem_size(dtype), st);
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}

}  // namespace

// SMs of the current device, queried once per device; -1 on error.
int sm_count() {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int count[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (count[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        count[dev] = v;
    }
    return count[dev];
}

// Grid size for the grid-stride kernels: one block per kThreads units, at
// most kWaves blocks per SM.
int grid_blocks(long long units) {
    const int sms = sm_count();
    if (sms < 1) return -1;
    const long long want = (units + kThreads - 1) / kThreads;
    const long long cap = (long long)sms * kWaves;
    const long long b = want < cap ? want : cap;
    return (int)(b < 1 ? 1 : b);
}

template <int ES>
cudaError_t launch_gather_es(const GatherParams& p_in, cudaStream_t st) {
    GatherParams p = p_in;
    const long long nvec = (p.M * ES + 15) / 16;
    const int slots = nvec * p.n >= kGatherWideVectors ? 8 : 2;
    const int blocks = grid_blocks((nvec + slots - 1) / slots);
    if (blocks < 1) return cudaErrorInvalidConfiguration;
    // Rank groups: double them while the grid is short of the target (8
    // blocks per SM for the wide blocks of 8 vectors a thread, 2 for blocks
    // of 2) and every group keeps at least 4 outputs (so the extra source
    // reads stay a quarter of the writes at most).  Measured: with 2 vectors
    // a target of 8 split 32 MiB x 8 ranks into two groups and cost 15 %;
    // with 8 vectors a target of 2 left 32 MiB x 64 ranks one group of 1024
    // blocks and cost 20 %.
    const int target = (slots == 8 ? 8 : 2) * sm_count();
    int groups = 1;
    while ((long long)blocks * groups < target && p.n / (groups * 2) >= 4) groups *= 2;
    p.rpg = (p.n + groups - 1) / groups;
    // programmatic dependent launch: the gather may be scheduled while the
    // preceding kernel drains; it waits on griddepcontrol before any access
    const dim3 grid(blocks, groups);
    // 2-byte shards off the 16-byte grid (shard s's vectors start s*q
    // elements into the index space, plus its base's own offset) take the
    // instances that realign their loads across the warp.
    if constexpr (ES == 2) {
        const long long shards = (p.M + p.q - 1) / p.q;
        bool realign = shards > 1 && (p.q * ES) % 16 != 0;
        for (long long s = 0; s < shards && !realign; ++s)
            realign = (reinterpret_cast<uintptr_t>(p.in[s]) & 15) != 0;
        if (realign) {
            if (slots == 8) return launch_pdl(vc_ag_kernel<ES, 8, true>, grid, dim3(kThreads), st, p);
            return launch_pdl(vc_ag_kernel<ES, 2, true>, grid, dim3(kThreads), st, p);
        }
    }
    if (slots == 8) return launch_pdl(vc_ag_kernel<ES, 8, false>, grid, dim3(kThreads), st, p);
    return launch_pdl(vc_ag_kernel<ES, 2, false>, grid, dim3(kThreads), st, p);
}

cudaError_t launch_gather(const GatherParams& p, int esize, cudaStream_t st) {
    switch (esize) {
    case 2: return launch_gather_es<2>(p, st);
    case 4: return launch_gather_es<4>(p, st);
    case 8: return launch_gather_es<8>(p, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vc

using namespace vc;

extern "C" {

size_t vc_shard_count(size_t count, int nranks) {
    if (nranks < 1) return 0;
    return count / (size_t)nranks + (count % (size_t)nranks != 0 ? 1 : 0);
}

vc_status_t vc_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int nranks,
                              size_t count, vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                              vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (!valid_op(op) || !valid_order(order)) return VC_ERR_INVALID_ARGUMENT;
    if (order == VC_ORDER_RECURSIVE_HALVING && !is_pow2(nranks)) return VC_ERR_UNSUPPORTED;
    if (count == 0) return VC_SUCCESS;
    if ((s = check_table(sendbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(recvbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_alias(sendbufs, bm, recvbufs, bq, nranks, false)) != VC_SUCCESS) return s;
    return launch_reduce(sendbufs, recvbufs, nranks, count, dtype, op, order, true,
                         static_cast<cudaStream_t>(stream));
}

vc_status_t vc_all_gather(const void* const* sendbufs, void* const* recvbufs, int nranks,
                          size_t count, vc_dtype_t dtype, vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (count == 0) return VC_SUCCESS;
    if ((s = check_table(sendbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(recvbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_alias(sendbufs, bq, recvbufs, bm, nranks, false)) != VC_SUCCESS) return s;
    return launch_all_gather(sendbufs, recvbufs, nranks, count, dtype,
                             static_cast<cudaStream_t>(stream));
}

vc_status_t vc_all_reduce(const void* const* sendbufs, void* const* recvbufs, int nranks,
                          size_t count, vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                          vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (!valid_op(op) || !valid_order(order)) return VC_ERR_INVALID_ARGUMENT;
    if (order == VC_ORDER_RECURSIVE_HALVING && !is_pow2(nranks)) return VC_ERR_UNSUPPORTED;
    if (count == 0) return VC_SUCCESS;
    if ((s = check_table(sendbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(recvbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_alias(sendbufs, bm, recvbufs, bm, nranks, true)) != VC_SUCCESS) return s;
    return launch_reduce(sendbufs, recvbufs, nranks, count, dtype, op, order, false,
                         static_cast<cudaStream_t>(stream));
}

vc_status_t vc_all_reduce_decomposed(const void* const* sendbufs, void* const* shardbufs,
                                     void* const* recvbufs, int nranks, size_t count,
                                     vc_dtype_t dtype, vc_op_t op, vc_order_t order,
                                     vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (!valid_op(op) || !valid_order(order)) return VC_ERR_INVALID_ARGUMENT;
    if (order == VC_ORDER_RECURSIVE_HALVING && !is_pow2(nranks)) return VC_ERR_UNSUPPORTED;
    if (count == 0) return VC_SUCCESS;
    if ((s = check_table(sendbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(shardbufs, nranks, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(recvbufs, nranks, dtype)) != VC_SUCCESS) return s;
    // shards overlap neither the inputs nor the outputs nor each other
    if ((s = check_alias(sendbufs, bm, shardbufs, bq, nranks, false)) != VC_SUCCESS) return s;
    if ((s = check_alias(const_cast<const void* const*>(recvbufs), bm, shardbufs, bq, nranks,
                         false)) != VC_SUCCESS)
        return s;
    if ((s = check_alias(sendbufs, bm, recvbufs, bm, nranks, true)) != VC_SUCCESS) return s;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    s = launch_reduce(sendbufs, shardbufs, nranks, count, dtype, op, order, true, st);
    if (s != VC_SUCCESS) return s;
    return launch_all_gather(const_cast<const void* const*>(shardbufs), recvbufs, nranks, count,
                             dtype, st);
}

vc_status_t vc_reduce(const void* const* sendbufs, void* recvbuf, int nranks, size_t count,
                      vc_dtype_t dtype, vc_op_t op, vc_order_t order, vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (!valid_op(op) || !valid_order(order)) return VC_ERR_INVALID_ARGUMENT;
    if (order == VC_ORDER_RECURSIVE_HALVING && !is_pow2(nranks)) return VC_ERR_UNSUPPORTED;
    if (count == 0) return VC_SUCCESS;
    if ((s = check_table(sendbufs, nranks, dtype)) != VC_SUCCESS) return s;
    void* const out[1] = {recvbuf};
    if ((s = check_table(out, 1, dtype)) != VC_SUCCESS) return s;
    // the output may be exactly one rank's input (in place at the root)
    const Range o = range_of(recvbuf, bm);
    for (int r = 0; r < nranks; ++r)
        if (overlap(o, range_of(sendbufs[r], bm)) && sendbufs[r] != recvbuf) return VC_ERR_ALIAS;
    int same = 0;
    for (int r = 0; r < nranks; ++r) same += (sendbufs[r] == recvbuf);
    if (same > 1) return VC_ERR_ALIAS;  // would be read as two ranks and written
    return launch_reduce(sendbufs, out, nranks, count, dtype, op, order, false,
                         static_cast<cudaStream_t>(stream), 1);
}

vc_status_t vc_broadcast(const void* sendbuf, void* const* recvbufs, int nranks, size_t count,
                         vc_dtype_t dtype, vc_stream_t stream) {
    size_t bm, bq;
    vc_status_t s = check_shape(nranks, count, dtype, &bm, &bq);
    if (s != VC_SUCCESS) return s;
    if (count == 0) return VC_SUCCESS;
    const void* const src[1] = {sendbuf};
    if ((s = check_table(src, 1, dtype)) != VC_SUCCESS) return s;
    if ((s = check_table(recvbufs, nranks, dtype)) != VC_SUCCESS) return s;
    // outputs pairwise disjoint; one of them may be the source itself (the
    // root's own buffer), which is then left as it is
    void* outs[VC_MAX_RANKS];
    int nout = 0;
    const Range in = range_of(sendbuf, bm);
    for (int r = 0; r < nranks; ++r) {
        const Range o = range_of(recvbufs[r], bm);
        for (int t = 0; t < r; ++t)
            if (overlap(o, range_of(recvbufs[t], bm))) return VC_ERR_ALIAS;
        if (recvbufs[r] == sendbuf) continue;
        if (overlap(o, in)) return VC_ERR_ALIAS;
        outs[nout++] = recvbufs[r];
    }
    return launch_broadcast(sendbuf, outs, nout, count, dtype, static_cast<cudaStream_t>(stream));
}

const char* vc_status_string(vc_status_t status) {
    switch (status) {
    case VC_SUCCESS: return "success";
    case VC_ERR_INVALID_ARGUMENT: return "invalid argument";
    case VC_ERR_UNSUPPORTED: return "unsupported: recursive halving needs a power-of-two rank count";
    case VC_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case VC_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
    }
}

}  // extern "C"
