// gdn_noalloc.cu -- gdn_backward_noalloc: the backward with its scratch memory in a
// fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the moment they run the
// backward -- code running under a memory budget that a host framework has already
// handed out in full, plugin or embedded hosts that expose no device allocator to their
// extensions, or call sites that must not trigger an allocator at all.  For them the
// scratch lives in one file-scope __device__ array of kNoAllocScratchBytes that every
// GPU which loads this library keeps until the process exits.
//
// Rules of use:
//   * The first call on a device (with that device current) looks up the array's device
//     address with cudaGetSymbolAddress; make that first call before any stream capture.
//   * Every call on a device shares the same array and leaves its contents behind.  The
//     backward writes every scratch element it reads within the same call, so nothing
//     has to start at zero, but two calls whose work overlaps on the GPU (different
//     streams, no ordering between them) race on the array and give wrong results.
//   * Problems whose workspace exceeds kNoAllocScratchBytes are rejected with
//     GDN_ERR_WORKSPACE before anything is launched.
//   * The looked-up address is kept for the life of the process.  A cudaDeviceReset
//     unloads the module that holds the array, so after one the address is stale: the
//     entry point is not for processes that reset a device they use it on.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" {

gdn_status_t gdn_backward_noalloc(const gdn_params_t* p, const void* q, const void* k,
                                  const void* v, const void* g, const void* beta,
                                  const float* ckpt, const void* gy, const float* dstate_T,
                                  float* packed_grads, void* stream)
{
    char msg[256];
    if (!p) {
        gdn::set_last_error("params is NULL");
        return GDN_ERR_INVALID_ARG;
    }
    const size_t need = gdn_backward_workspace_bytes(p);
    if (need > kNoAllocScratchBytes) {
        snprintf(msg, sizeof msg,
                 "problem needs %zu bytes of backward scratch; the no-allocation entry point "
                 "holds %zu bytes per device (use gdn_backward with a caller workspace)",
                 need, kNoAllocScratchBytes);
        gdn::set_last_error(msg);
        return GDN_ERR_WORKSPACE;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaGetDevice failed: %s", cudaGetErrorString(e));
        gdn::set_last_error(msg);
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof msg,
                 "device %d is beyond the %d devices the no-allocation entry point keeps a "
                 "scratch address for", dev, kMaxDevices);
        gdn::set_last_error(msg);
        return GDN_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess || !addr) {
                snprintf(msg, sizeof msg, "cudaGetSymbolAddress failed: %s",
                         cudaGetErrorString(e));
                gdn::set_last_error(msg);
                return GDN_ERR_CUDA;
            }
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    return gdn_backward(p, q, k, v, g, beta, ckpt, gy, dstate_T, packed_grads, scratch,
                        kNoAllocScratchBytes, stream);
}

}  // extern "C"
