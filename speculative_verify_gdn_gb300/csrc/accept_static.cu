// accept_static.cu — spec_accept_static: spec_accept for callers that cannot allocate device memory.
//
// spec_accept needs a caller-provided device workspace. Some callers have no way to get one: code
// running where cudaMalloc is not permitted or not available to it (inside a host callback, in a
// plug-in that only receives device pointers from its host framework, in a process whose memory
// pool is fixed up front), or code that must not allocate on the hot path at all. For them this
// entry point uses a fixed scratch array that lives in the library's own device memory image:
// it is a file-scope __device__ array, created when the library's module is loaded on a device
// and held by that device until the process exits. Nothing here calls cudaMalloc or cudaFree.
//
// Limits and sharing:
//  - The scratch holds GDN_STATIC_SCRATCH_BYTES bytes; a call that needs more (see
//    spec_workspace_bytes) is rejected with GDN_ERR_UNSUPPORTED and a message.
//  - Every call on a device uses the same array and leaves its contents behind. The accept kernels
//    write every scratch word they read before reading it, so nothing has to start at zero, but two
//    calls whose kernels overlap on the GPU (different streams, no ordering) race on the array.
//  - The first call on each device looks up the array's device address (cudaGetSymbolAddress with
//    that device current) and keeps it for that device's current context; a call made after the
//    context changed (cudaDeviceReset reloads the module, possibly at another address) looks it up
//    again. Make the first call on a device, and the first after a reset, outside of any stream
//    capture.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdnspec.h"
#include "kernels.h"

namespace {

__device__ __align__(256) unsigned char g_accept_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long ctx;   // context the address belongs to (gdn::current_context_id)
    void* addr;
};
std::mutex g_mu;
ScratchAddr g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the current device's current context.
int scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return gdn::report_error(GDN_ERR_CUDA, "spec_accept_static: cudaGetDevice failed: %s",
                                 cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return gdn::report_error(GDN_ERR_UNSUPPORTED, "spec_accept_static: device %d", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long ctx = gdn::current_context_id();
    ScratchAddr& slot = g_scratch[dev];
    if (!slot.addr || !ctx || slot.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_accept_scratch);
        if (e != cudaSuccess || !p)
            return gdn::report_error(GDN_ERR_CUDA,
                                     "spec_accept_static: cudaGetSymbolAddress failed: %s",
                                     cudaGetErrorString(e));
        // the lookup makes the device's primary context current if none was
        slot.ctx = ctx ? ctx : gdn::current_context_id();
        slot.addr = p;
    }
    *out = slot.addr;
    return GDN_OK;
}

}  // namespace

extern "C" int spec_accept_static(const spec_dims* d, const void* logits, const int32_t* drafts,
                                  int32_t mode, float temperature, uint64_t seed, uint64_t round,
                                  int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                                  void* stream) {
    const int32_t eff = (mode == SPEC_MODE_SAMPLE && !(temperature > 0.f)) ? SPEC_MODE_GREEDY : mode;
    const size_t need = spec_workspace_bytes(d, eff);
    if (need == 0) {
        // invalid shape or mode: let spec_accept report it with its own message
        return spec_accept(d, logits, drafts, mode, temperature, seed, round, nullptr, 0, n_acc,
                           out_tokens, status, stream);
    }
    if (need > size_t(GDN_STATIC_SCRATCH_BYTES))
        return gdn::report_error(GDN_ERR_UNSUPPORTED,
                                 "spec_accept_static: this shape needs %zu bytes of scratch, the "
                                 "static scratch holds %zu; call spec_accept with a workspace",
                                 need, size_t(GDN_STATIC_SCRATCH_BYTES));
    void* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    return spec_accept(d, logits, drafts, mode, temperature, seed, round, scratch,
                       size_t(GDN_STATIC_SCRATCH_BYTES), n_acc, out_tokens, status, stream);
}
