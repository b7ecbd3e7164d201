// rollback.cu — gdn_rollback / gdn_rollback_path: tape-replay rollback (sm_103a).
//
// "Speculative Decoding on GDN Hybrid Architectures: A 31-Experiment Investigation", §4
// (Tape-Replay 回滚): after a partial acceptance of n of the T verified positions, restore the
// pre-verify snapshot and replay only the accepted steps, state = state·g[t] + δ[t] k[t]ᵀ for
// t < n, at cost O(n); rebuild the conv state from the last (W−1) raw qkv rows.
//
// Here the snapshot is the state buffer itself (verify never writes it), so "restore" is free and
// the replay of n steps is folded into one pass over the state:
//     S_n = Γ_total · S_0 + Σ_{s<n} (Γ_{s+1..n-1} δ_s) k_sᵀ,   Γ_total = Π_{s<n} g_s,
// which reads and writes each state element once (HBM-bound) with n+1 FMAs per element.
// The state is row-major S ([i][j], j contiguous): lanes own consecutive key columns j (16-byte
// accesses, coalesced rows), warps own rows i. One 256-thread CTA per (layer, sequence, value
// head); n is read on the device, so a CTA whose sequence accepted nothing exits at once and the
// whole call needs no host synchronisation.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

template <int RPL>
__device__ __forceinline__ void ld_rows_cs(const float* p, float (&v)[RPL]) {
    if constexpr (RPL == 4) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else if constexpr (RPL == 2) {
        const float2 x = __ldcs(reinterpret_cast<const float2*>(p));
        v[0] = x.x; v[1] = x.y;
    } else {
        v[0] = __ldcs(p);
    }
}

template <int RPL>
__device__ __forceinline__ void st_rows_cs(float* p, const float (&v)[RPL]) {
    if constexpr (RPL == 4) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    } else if constexpr (RPL == 2) {
        __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
    } else {
        __stcs(p, v[0]);
    }
}

template <typename IO, int D, int NMAX, bool PATH>
__global__ void __launch_bounds__(256, (NMAX <= 8 ? 2 : 1))
gdn_rollback_kernel(const RollbackArgs a) {
    constexpr int CPL = D / 32;      // consecutive key columns j per lane
    constexpr int NW = 8;            // warps; warp w owns state rows i = w, w + 8, ...
    constexpr int RPW = D / NW;
    __shared__ float Ds[NMAX][D];    // scaled innovations δ'_s[i] = Γ_{s+1..n-1} δ_s[i]
    __shared__ float coef[NMAX];
    __shared__ float gs[NMAX];
    __shared__ int nodes[NMAX];
    __shared__ float gtot;
    __shared__ int bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
    const int T = a.T, Hv = a.Hv, Hk = a.Hk, C = a.C, W = a.W;
    const int kh = h / (Hv / Hk);
    const size_t lb = size_t(l) * a.B + b;

    const int n = __ldg(a.n_acc + b);
    const int cap = PATH ? (a.P < T ? a.P : T) : T;
    if (n < 0 || n > cap) {
        if (tid == 0 && h == 0 && l == 0) set_status(a.status, GDN_STATUS_BAD_NACC);
        return;
    }
    if (n == 0) return;              // the snapshot is still in place

    // every load is issued before the first wait: the state slice of this thread, the gates, the
    // tape rows (chains: rows 0 .. n-1; paths: the path's nodes, read by every thread, clamped to
    // a valid row until the check below)
    float* S = a.state + (lb * Hv + h) * size_t(D) * D;   // row-major S: [i][j]
    const int j0 = lane * CPL;
    float v[RPW][CPL];
#pragma unroll
    for (int u = 0; u < RPW; ++u) ld_rows_cs<CPL>(S + size_t(warp + NW * u) * D + j0, v[u]);

    if (tid == 0) bad = 0;
    auto node_of = [&](int s2) -> int {
        if (!PATH) return s2;
        const int nd = __ldg(a.path + size_t(b) * a.P + s2);
        return (nd >= 0 && nd < T) ? nd : -1;
    };
    float gv = 0.f;
    int my_node = 0;
    if (tid < n) {
        my_node = node_of(tid);
        gv = __ldg(a.g + (lb * T + (my_node < 0 ? 0 : my_node)) * Hv + h);
    }
    float kr[NMAX][CPL];   // k_s[j0 .. j0+CPL) of this lane's columns
#pragma unroll
    for (int s = 0; s < NMAX; ++s) {
#pragma unroll
        for (int r = 0; r < CPL; ++r) kr[s][r] = 0.f;
        if (s < n) {
            const int nd = node_of(s);
            const float* src = a.tape_k + ((lb * T + (nd < 0 ? 0 : nd)) * Hk + kh) * size_t(D) + j0;
#pragma unroll
            for (int r = 0; r < CPL; ++r) kr[s][r] = __ldg(src + r);
        }
    }
    for (int idx = tid; idx < n * D; idx += 256) {       // raw δ_s[i]; Γ_{s+1..n-1} applied below
        const int s2 = idx / D, i = idx - s2 * D;
        const int nd = node_of(s2);
        Ds[s2][i] = __ldg(a.tape_delta + ((lb * T + (nd < 0 ? 0 : nd)) * Hv + h) * size_t(D) + i);
    }
    __syncthreads();
    if (tid < n) {
        nodes[tid] = my_node < 0 ? 0 : my_node;
        gs[tid] = gv;
        if (my_node < 0) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (bad) {
        if (tid == 0 && h == 0 && l == 0) set_status(a.status, GDN_STATUS_BAD_PATH);
        return;
    }
    if (tid == 0) {
        float c = 1.f;
        for (int s2 = n - 1; s2 >= 0; --s2) {
            coef[s2] = c;                                  // Γ_{s+1..n-1}
            c *= gs[s2];
        }
        gtot = c;                                          // Γ_{0..n-1}
    }
    __syncthreads();
    const float G = gtot;

    // S_n[i][j] = Γ_total S_0[i][j] + Σ_s Γ_{s+1..n-1} δ_s[i] k_s[j]
#pragma unroll
    for (int u = 0; u < RPW; ++u) {
        const int i = warp + NW * u;
#pragma unroll
        for (int r = 0; r < CPL; ++r) v[u][r] *= G;
#pragma unroll
        for (int s2 = 0; s2 < NMAX; ++s2) {
            if (s2 < n) {
                const float d = coef[s2] * Ds[s2][i];
#pragma unroll
                for (int r = 0; r < CPL; ++r) v[u][r] = fmaf(d, kr[s2][r], v[u][r]);
            }
        }
        st_rows_cs<CPL>(S + size_t(i) * D + j0, v[u]);
    }

    // conv state: last W-1 rows of (conv_state ++ accepted raw rows); channels split over heads
    const int cper = (C + Hv - 1) / Hv;
    const int c_lo = h * cper, c_hi = min(C, c_lo + cper);
    IO* cs = static_cast<IO*>(a.conv_state) + lb * size_t(W - 1) * C;
    const IO* x = static_cast<const IO*>(a.qkv) + lb * size_t(T) * C;
    for (int c = c_lo + tid; c < c_hi; c += 256) {
        IO vals[3];
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            if (r < W - 1) {
                const int q = n + r;   // index in the combined sequence
                vals[r] = (q < W - 1) ? cs[size_t(q) * C + c]
                                      : x[size_t(nodes[q - (W - 1)]) * C + c];
            }
        }
#pragma unroll
        for (int r = 0; r < 3; ++r)
            if (r < W - 1) cs[size_t(r) * C + c] = vals[r];
    }
}

template <typename IO, int D, int NMAX, bool PATH>
static cudaError_t launch_rb(const RollbackArgs& a, cudaStream_t s) {
    dim3 grid(a.Hv, a.B, a.L);
    gdn_rollback_kernel<IO, D, NMAX, PATH><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename IO, bool PATH>
static cudaError_t launch_rb_io(const RollbackArgs& a, int D, cudaStream_t s) {
    const int cap = PATH ? (a.P < a.T ? a.P : a.T) : a.T;
    const int nm = cap <= 4 ? 4 : cap <= 8 ? 8 : cap <= 16 ? 16 : 32;
#define GDN_R_CASE(DD, NM) \
    if (D == DD && nm == NM) return launch_rb<IO, DD, NM, PATH>(a, s);
    GDN_R_CASE(32, 4) GDN_R_CASE(32, 8) GDN_R_CASE(32, 16) GDN_R_CASE(32, 32)
    GDN_R_CASE(64, 4) GDN_R_CASE(64, 8) GDN_R_CASE(64, 16) GDN_R_CASE(64, 32)
    GDN_R_CASE(128, 4) GDN_R_CASE(128, 8) GDN_R_CASE(128, 16) GDN_R_CASE(128, 32)
#undef GDN_R_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_rollback(const RollbackArgs& a, int D, int io_dtype, cudaStream_t s) {
    const bool path = a.path != nullptr;
    if (io_dtype == GDN_DTYPE_BF16)
        return path ? launch_rb_io<__nv_bfloat16, true>(a, D, s)
                    : launch_rb_io<__nv_bfloat16, false>(a, D, s);
    return path ? launch_rb_io<float, true>(a, D, s) : launch_rb_io<float, false>(a, D, s);
}

}  // namespace gdn
