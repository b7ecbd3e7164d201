// host_util.cu — host-side launch helpers shared by the kernels' launchers.
//
// Per-kernel attributes such as the dynamic shared-memory opt-in belong to one (context, kernel)
// pair: a process that drives two GPUs, or that resets a device (which creates a new primary
// context and reloads the library's module), must set them again. The helpers here therefore key
// what they remember on the current context's unique id (cuCtxGetId, fetched from the driver
// through the runtime, so the library still links no libcuda), and update it under a mutex so
// that the recorded size is always one that was actually set.
#include <cuda.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"

namespace gdn {
namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        p = nullptr;
    return reinterpret_cast<Fn>(p);
}

std::mutex g_mu;
std::map<std::pair<unsigned long long, const void*>, size_t> g_optin;   // (context, kernel) -> bytes
std::map<int, int> g_nsm;                                                // device -> SM count

}  // namespace

unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_cur || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id + 1;   // 0 stays "unknown"
}

cudaError_t smem_optin(const void* kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;   // within the default limit: nothing to set
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long ctx = current_context_id();
    if (ctx) {
        auto it = g_optin.find({ctx, kernel});
        if (it != g_optin.end() && it->second >= bytes) return cudaSuccess;
    }
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e != cudaSuccess) return e;
    // the call above made the device's primary context current if none was: key on it now
    const unsigned long long ctx_now = ctx ? ctx : current_context_id();
    if (ctx_now) g_optin[{ctx_now, kernel}] = bytes;
    return cudaSuccess;
}

cudaError_t device_sm_count(int* n) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_nsm.find(dev);
    if (it != g_nsm.end()) {
        *n = it->second;
        return cudaSuccess;
    }
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_nsm[dev] = v;
    *n = v;
    return cudaSuccess;
}

}  // namespace gdn
