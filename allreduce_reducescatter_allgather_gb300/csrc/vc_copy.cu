// vc_copy_tiles: many independent byte ranges copied in one launch -- the
// packing of small gradient tensors into a bucket buffer and back.
#include "vc.h"
#include "vc_device.cuh"

namespace vc {
namespace {

// One block per tile (grid-stride over tiles).  Each thread moves up to four
// 16-byte vectors per round, all loaded before any is stored; unaligned
// tiles fall back to 4-byte or 1-byte units.
__global__ void __launch_bounds__(kThreads) vc_copy_tiles_kernel(const vc_copy_tile_t* tiles,
                                                                  int ntiles) {
    constexpr int S = 4;
    // launched with programmatic stream serialization: wait for the kernel
    // before this one to complete (and its writes to be visible) first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const vc_copy_tile_t tile = tiles[t];
        const unsigned char* src = static_cast<const unsigned char*>(tile.src);
        unsigned char* dst = static_cast<unsigned char*>(tile.dst);
        const size_t bytes = tile.bytes;
        const uintptr_t mis = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
        if ((mis & 15) == 0 && (bytes & 15) == 0) {
            const size_t nv = bytes / 16;
            const uint4* s = reinterpret_cast<const uint4*>(src);
            uint4* d = reinterpret_cast<uint4*>(dst);
            for (size_t v0 = threadIdx.x; v0 < nv; v0 += (size_t)blockDim.x * S) {
                uint4 buf[S];
#pragma unroll
                for (int u = 0; u < S; ++u) {
                    const size_t v = v0 + (size_t)u * blockDim.x;
                    if (v < nv) buf[u] = s[v];
                }
#pragma unroll
                for (int u = 0; u < S; ++u) {
                    const size_t v = v0 + (size_t)u * blockDim.x;
                    if (v < nv) d[v] = buf[u];
                }
            }
        } else if ((mis & 3) == 0 && (bytes & 3) == 0) {
            const unsigned* s = reinterpret_cast<const unsigned*>(src);
            unsigned* d = reinterpret_cast<unsigned*>(dst);
            for (size_t k = threadIdx.x; k < bytes / 4; k += blockDim.x) d[k] = s[k];
        } else {
            for (size_t k = threadIdx.x; k < bytes; k += blockDim.x) dst[k] = src[k];
        }
    }
    // this block is done: a kernel launched after this one may start
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace
}  // namespace vc

using namespace vc;

extern "C" vc_status_t vc_copy_tiles(const vc_copy_tile_t* dev_tiles, int ntiles,
                                     vc_stream_t stream) {
    if (ntiles < 0) return VC_ERR_INVALID_ARGUMENT;
    if (ntiles == 0) return VC_SUCCESS;
    if (dev_tiles == nullptr || (reinterpret_cast<uintptr_t>(dev_tiles) & 7) != 0)
        return VC_ERR_INVALID_ARGUMENT;
    const char* hook = getenv("VC_TEST_FAIL_LAUNCH");
    if (hook != nullptr && hook[0] != '\0' && hook[0] != '0') return VC_ERR_CUDA;
    const int blocks = grid_blocks((long long)ntiles * kThreads);
    if (blocks < 1) return VC_ERR_CUDA;
    const cudaError_t e = launch_pdl(vc_copy_tiles_kernel, dim3(blocks), dim3(kThreads),
                                     static_cast<cudaStream_t>(stream), dev_tiles, ntiles);
    return e == cudaSuccess ? VC_SUCCESS : VC_ERR_CUDA;
}
