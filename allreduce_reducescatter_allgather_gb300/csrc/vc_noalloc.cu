// vc_all_reduce_decomposed_noalloc: the decomposed AllReduce for callers that
// cannot allocate device memory.
//
// The N intermediate shards, which vc_all_reduce_decomposed takes from the
// caller, live here in one file-scope device array of a fixed size.  This
// file holds no kernel, so the array is the only content of its device-code
// module: under lazy module loading it is placed on a device at the first
// call there (the cudaGetSymbolAddress below), eagerly when the context is
// set up otherwise, and held until the process exits.  The call itself
// allocates nothing: it looks up the array's device address once per device,
// carves it into N shards and launches the same ReduceScatter and AllGather
// kernels as the other entry points.  The cached address does not survive a
// cudaDeviceReset of its device.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "vc.h"
#include "vc_device.cuh"

namespace vc {
namespace {

// The shared shard scratch.  In host code this name is only a stand-in for
// the device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char noalloc_scratch[VC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
constexpr size_t kShardAlign = 256;  // every shard starts on a 256-byte boundary

std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on
// the first call on each device, with that device current.
vc_status_t scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return VC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return VC_SUCCESS;
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

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, const void* b, size_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bytes && y < x + bytes;
}

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" vc_status_t vc_all_reduce_decomposed_noalloc(const void* const* sendbufs,
                                                         void* const* recvbufs, int nranks,
                                                         size_t count, vc_dtype_t dtype,
                                                         vc_op_t op, vc_order_t order,
                                                         vc_stream_t stream) {
    if (nranks < 1 || nranks > VC_MAX_RANKS) return VC_ERR_INVALID_ARGUMENT;
    const int es = esize(dtype);
    if (es == 0 || op < VC_SUM || op > VC_AVG) return VC_ERR_INVALID_ARGUMENT;
    if (order < VC_ORDER_RING || order > VC_ORDER_DOUBLE_BINARY_TREE) return VC_ERR_INVALID_ARGUMENT;
    if (order == VC_ORDER_RECURSIVE_HALVING && (nranks & (nranks - 1)) != 0) return VC_ERR_UNSUPPORTED;
    if (count == 0) return VC_SUCCESS;
    // the shards must fit the fixed scratch: N shards of q elements, each
    // rounded up to 256 bytes
    if (count > VC_NOALLOC_SCRATCH_BYTES) return VC_ERR_INVALID_ARGUMENT;
    const size_t q = vc_shard_count(count, nranks);
    const size_t stride = (q * (size_t)es + kShardAlign - 1) / kShardAlign * kShardAlign;
    if (stride * (size_t)nranks > VC_NOALLOC_SCRATCH_BYTES) return VC_ERR_INVALID_ARGUMENT;
    if (sendbufs == nullptr || recvbufs == nullptr) return VC_ERR_INVALID_ARGUMENT;
    const size_t bytes = count * (size_t)es;
    for (int r = 0; r < nranks; ++r) {
        if (sendbufs[r] == nullptr || recvbufs[r] == nullptr) return VC_ERR_INVALID_ARGUMENT;
        if (!aligned(sendbufs[r], es) || !aligned(recvbufs[r], es)) return VC_ERR_INVALID_ARGUMENT;
    }
    // outputs: pairwise disjoint, and disjoint from every input except their
    // own (in place)
    for (int r = 0; r < nranks; ++r) {
        for (int s = 0; s < nranks; ++s) {
            if (s != r && overlaps(recvbufs[r], recvbufs[s], bytes)) return VC_ERR_ALIAS;
            if (overlaps(recvbufs[r], sendbufs[s], bytes) &&
                !(s == r && recvbufs[r] == sendbufs[s]))
                return VC_ERR_ALIAS;
        }
    }
    void* base = nullptr;
    vc_status_t st = scratch_address(&base);
    if (st != VC_SUCCESS) return st;

    ReduceParams rp;
    memset(&rp, 0, sizeof rp);
    GatherParams gp;
    memset(&gp, 0, sizeof gp);
    bool in_vec = true, out_vec = true;
    for (int r = 0; r < nranks; ++r) {
        void* shard = static_cast<unsigned char*>(base) + (size_t)r * stride;
        rp.in[r] = sendbufs[r];
        rp.out[r] = shard;
        gp.in[r] = shard;
        gp.out[r] = recvbufs[r];
        in_vec = in_vec && aligned(sendbufs[r], 16);
        out_vec = out_vec && aligned(recvbufs[r], 16);
    }
    rp.M = gp.M = (long long)count;
    rp.q = gp.q = (long long)q;
    rp.limit = (long long)nranks * (long long)q;
    rp.half = ((long long)count + 1) / 2;
    rp.inv_q = gp.inv_q = 1.0f / (float)q;
    rp.n = gp.n = nranks;
    rp.nout = nranks;
    rp.avg = (op == VC_AVG);
    rp.vec_ok = in_vec;
    gp.vec_ok = out_vec;

    const char* hook = getenv("VC_TEST_FAIL_LAUNCH");
    if (hook != nullptr && hook[0] != '\0' && hook[0] != '0') return VC_ERR_CUDA;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (dtype) {
    case VC_INT32: e = launch_reduce_i32(rp, (int)op, (int)order, true, cs); break;
    case VC_INT64: e = launch_reduce_i64(rp, (int)op, (int)order, true, cs); break;
    case VC_FLOAT32: e = launch_reduce_f32(rp, (int)op, (int)order, true, cs); break;
    default: e = launch_reduce_bf16(rp, (int)op, (int)order, true, cs); break;
    }
    if (e != cudaSuccess) return VC_ERR_CUDA;
    e = launch_gather(gp, es, cs);
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}
