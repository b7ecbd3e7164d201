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
// With one gate per key channel (g [B, T, Hv, Dk]) the products are per column j: Γ_total[j]
// scales column j of S_0 and k_s[j] carries Π_{s<r<n} a_r[j]; the pass is otherwise the same.
// The state is row-major S ([i][j], j contiguous). One 256-thread CTA per (layer, sequence, value
// head) moves its slice by bulk copy into shared memory and back (64 KiB at d = 128, so three
// CTAs per SM keep ~200 KiB of state in flight; registers would hold two); lanes own consecutive
// key columns j, warps own rows i. n is read on the device, so a CTA whose sequence accepted
// nothing exits at once and the whole call needs no host synchronisation.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

// shared memory of one CTA: the state slice [D][D], then δ_s [NMAX][D] and k_s [NMAX][D]
template <int D, int NMAX>
struct RbSmem {
    static constexpr size_t SLICE = size_t(D) * D * 4, CHUNK = SLICE < 16384 ? SLICE : 16384;
    static constexpr size_t OFF_D = SLICE, OFF_K = OFF_D + size_t(NMAX) * D * 4;
    static constexpr size_t BYTES = OFF_K + size_t(NMAX) * D * 4;
    static_assert(SLICE % CHUNK == 0 && CHUNK % 16 == 0, "bulk-copy chunks");
};

template <typename IO, int D, int NMAX, bool PATH>
__global__ void __launch_bounds__(256)
gdn_rollback_kernel(const RollbackArgs a) {
    using Sm = RbSmem<D, NMAX>;
    constexpr int CPL = D / 32;      // consecutive key columns j per lane
    constexpr int NW = 8;            // warps; warp w owns state rows i = w, w + 8, ...
    constexpr int RPW = D / NW;
    extern __shared__ __align__(128) unsigned char rb_smem[];
    float* Sl = reinterpret_cast<float*>(rb_smem);                    // state slice S_0 -> S_n
    float (*Ds)[D] = reinterpret_cast<float (*)[D]>(rb_smem + Sm::OFF_D);   // innovations δ_s[i]
    float (*Ks)[D] = reinterpret_cast<float (*)[D]>(rb_smem + Sm::OFF_K);   // keys k_s[j]
    __shared__ float coef[NMAX];
    __shared__ float gs[NMAX];
    __shared__ int nodes[NMAX];
    __shared__ float gtot;
    __shared__ float gcol[D];        // per-key-channel gates: Γ_total per column j
    __shared__ int bad, load_ok;
    __shared__ __align__(8) uint64_t bar;

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

    // the state slice streams into shared memory by bulk copy while the tape is read: every load
    // is issued before the first wait (paths: the path's nodes are read by every thread, clamped
    // to a valid row until the check below)
    float* S = a.state + (lb * Hv + h) * size_t(D) * D;   // row-major S: [i][j]
    if (tid == 0) {
        bad = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar, uint32_t(Sm::SLICE));
#pragma unroll 1
        for (size_t o = 0; o < Sm::SLICE; o += Sm::CHUNK)
            bulk_g2s(rb_smem + o, reinterpret_cast<const unsigned char*>(S) + o, uint32_t(Sm::CHUNK), &bar);
    }
    auto node_of = [&](int s2) -> int {
        if (!PATH) return s2;
        const int nd = __ldg(a.path + size_t(b) * a.P + s2);
        return (nd >= 0 && nd < T) ? nd : -1;
    };
    float gv = 0.f;
    int my_node = 0;
    if (tid < n) {
        my_node = node_of(tid);
        gv = a.gate_dk ? 1.f : __ldg(a.g + (lb * T + (my_node < 0 ? 0 : my_node)) * Hv + h);
    }
    for (int idx = tid; idx < n * D; idx += 256) {       // raw δ_s[i] (Γ_{s+1..n-1} applied below), k_s[j]
        const int s2 = idx / D, i = idx - s2 * D;
        const int nd = node_of(s2), row = nd < 0 ? 0 : nd;
        Ds[s2][i] = __ldg(a.tape_delta + ((lb * T + row) * Hv + h) * size_t(D) + i);
        Ks[s2][i] = __ldg(a.tape_k + ((lb * T + row) * Hk + kh) * size_t(D) + i);
    }
    __syncthreads();
    if (tid < n) {
        nodes[tid] = my_node < 0 ? 0 : my_node;
        gs[tid] = gv;
        if (my_node < 0) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (a.gate_dk && tid < D) {      // column j = tid: k_s[j] *= Π_{s<r<n} a_r[j], Γ_total[j]
        const int j = tid;
        float av[NMAX];
#pragma unroll
        for (int s2 = 0; s2 < NMAX; ++s2)
            av[s2] = s2 < n ? __ldg(a.g + ((lb * T + nodes[s2]) * Hv + h) * size_t(D) + j) : 1.f;
        float c = 1.f;
#pragma unroll
        for (int s2 = NMAX - 1; s2 >= 0; --s2) {
            if (s2 < n) {
                Ks[s2][j] *= c;
                c *= av[s2];
            }
        }
        gcol[j] = c;
    }
    if (tid == 0) {
        float c = 1.f;
        for (int s2 = n - 1; s2 >= 0; --s2) {
            coef[s2] = c;                                  // Γ_{s+1..n-1}
            c *= gs[s2];
        }
        gtot = c;                                          // Γ_{0..n-1}
        // the slice must land before this CTA may leave, whatever happens below
        load_ok = mbar_wait_bounded(&bar, 0) ? 1 : 0;
        if (!load_ok) {
            set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
            mbar_wait_bounded(&bar, 0);
        }
    }
    __syncthreads();
    if (!load_ok || bad) {
        if (bad && tid == 0 && h == 0 && l == 0) set_status(a.status, GDN_STATUS_BAD_PATH);
        return;
    }
    mbar_try_wait(&bar, 0);          // completed: each thread observes the slice
    const int j0 = lane * CPL;
    float G[CPL];                    // Γ_total of this lane's columns
#pragma unroll
    for (int r = 0; r < CPL; ++r) G[r] = a.gate_dk ? gcol[j0 + r] : gtot;

    // S_n[i][j] = Γ_total S_0[i][j] + Σ_s Γ_{s+1..n-1} δ_s[i] k_s[j], in place in shared memory
    float kr[NMAX <= 8 ? NMAX : 1][CPL];
    if constexpr (NMAX <= 8) {
#pragma unroll
        for (int s2 = 0; s2 < NMAX; ++s2)
#pragma unroll
            for (int r = 0; r < CPL; ++r) kr[s2][r] = s2 < n ? Ks[s2][j0 + r] : 0.f;
    }
#pragma unroll 4
    for (int u = 0; u < RPW; ++u) {
        const int i = warp + NW * u;
        float v[CPL];
        if constexpr (CPL == 4) {
            const float4 x4 = *reinterpret_cast<const float4*>(Sl + i * D + j0);
            v[0] = G[0] * x4.x; v[1] = G[1] * x4.y; v[2] = G[2] * x4.z; v[3] = G[3] * x4.w;
        } else {
#pragma unroll
            for (int r = 0; r < CPL; ++r) v[r] = G[r] * Sl[i * D + j0 + r];
        }
        if constexpr (NMAX <= 8) {
#pragma unroll
            for (int s2 = 0; s2 < NMAX; ++s2) {
                const float d = s2 < n ? coef[s2] * Ds[s2][i] : 0.f;
#pragma unroll
                for (int r = 0; r < CPL; ++r) v[r] = fmaf(d, kr[s2][r], v[r]);
            }
        } else {
#pragma unroll 1
            for (int s2 = 0; s2 < n; ++s2) {
                const float d = coef[s2] * Ds[s2][i];
#pragma unroll
                for (int r = 0; r < CPL; ++r) v[r] = fmaf(d, Ks[s2][j0 + r], v[r]);
            }
        }
        if constexpr (CPL == 4) {
            *reinterpret_cast<float4*>(Sl + i * D + j0) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int r = 0; r < CPL; ++r) Sl[i * D + j0 + r] = v[r];
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the bulk store reads them
    __syncthreads();
    if (tid == 0) {
#pragma unroll 1
        for (size_t o = 0; o < Sm::SLICE; o += Sm::CHUNK)
            bulk_s2g(reinterpret_cast<unsigned char*>(S) + o, rb_smem + o, uint32_t(Sm::CHUNK));
        bulk_commit();
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
    if (tid == 0) bulk_wait_read_all();   // the slice stays until the store has read it
}

template <typename IO, int D, int NMAX, bool PATH>
static cudaError_t launch_rb(const RollbackArgs& a, cudaStream_t s) {
    constexpr size_t SMEM = RbSmem<D, NMAX>::BYTES;
    auto kern = gdn_rollback_kernel<IO, D, NMAX, PATH>;
    const cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hv, a.B, a.L);
    kern<<<grid, 256, SMEM, s>>>(a);
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
