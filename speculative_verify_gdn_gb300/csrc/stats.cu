// stats.cu — spec_stats_accumulate: acceptance counters for an adaptive speculation switch
// (colibrì ch.08 §4.1, adaptive off-switch: proposed and accepted draft totals, here with the
// histogram of accepted lengths). Integer atomics, so the totals are exact and order-free.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

constexpr int kStatThreads = 256;
constexpr int kStatMaxN = 64;      // histogram bins held in shared memory (N + 1 <= 65)

__global__ void __launch_bounds__(kStatThreads) spec_stats_kernel(int B, int N, const int32_t* n_acc,
                                                                  unsigned long long* stats,
                                                                  uint32_t* status) {
    __shared__ unsigned long long hist[kStatMaxN + 1];
    __shared__ unsigned long long acc;
    for (int k = threadIdx.x; k <= N; k += kStatThreads) hist[k] = 0ull;
    if (threadIdx.x == 0) acc = 0ull;
    __syncthreads();
    bool bad = false;
    for (int b = blockIdx.x * kStatThreads + threadIdx.x; b < B; b += gridDim.x * kStatThreads) {
        const int n = __ldg(n_acc + b);
        if (n < 0 || n > N) { bad = true; continue; }
        atomicAdd(&hist[n], 1ull);
        atomicAdd(&acc, static_cast<unsigned long long>(n));
    }
    if (bad) set_status(status, GDN_STATUS_BAD_NACC);
    __syncthreads();
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0)
            atomicAdd(&stats[0], static_cast<unsigned long long>(B) * static_cast<unsigned long long>(N));
        atomicAdd(&stats[1], acc);
    }
    for (int k = threadIdx.x; k <= N; k += kStatThreads)
        if (hist[k]) atomicAdd(&stats[2 + k], hist[k]);
}

cudaError_t launch_spec_stats(int B, int N, const int32_t* n_acc, uint64_t* stats, uint32_t* status,
                              cudaStream_t s) {
    int grid = (B + kStatThreads - 1) / kStatThreads;
    if (grid > 64) grid = 64;
    spec_stats_kernel<<<grid, kStatThreads, 0, s>>>(B, N, n_acc,
                                                    reinterpret_cast<unsigned long long*>(stats),
                                                    status);
    return cudaGetLastError();
}

}  // namespace gdn
