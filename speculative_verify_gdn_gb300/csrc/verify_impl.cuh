// verify_impl.cuh — gdn_verify / gdn_verify_tree kernel (sm_103a, tcgen05 tensor cores).
//
// What it computes (per layer l, sequence b, value head h; "GDN investigation" = "Speculative
// Decoding on GDN Hybrid Architectures: A 31-Experiment Investigation", §2.1, §2.2, §4):
//   conv + SiLU over each position's window, q/k L2-normalised per head, then the gated delta
//   rule u = g S k, δ = β (v − u), S ← g S + δ kᵀ, o = scale · S q, from the snapshot S_0,
//   node by node (chain: node t's parent is t−1; tree: an explicit parent array).
//   Writes o, the tape (δ per value head, normalised k per key head). S_0 is never written.
//   Chains and trees also take one gate per key channel (g [B, T, Hv, Dk], §4's tape layout):
//   S ← S·diag(a_t) + δ kᵀ with u = S·diag(a_t)·k; then the dense product reads the decayed
//   columns A_t ⊙ k_t, A_t ⊙ q_t (A_t: the gates of t and its ancestors) and the Gram block
//   carries the per-channel decays between each node and its ancestors.
//
// How (GB300 design):
//   * The state update is never materialised. With Γ(a→p) the product of the gates strictly
//     after node a up to node p on the path, the parent state of node v satisfies
//         S_p k_v = Γ(root→p) S_0 k_v + Σ_{a ∈ path(p)} Γ(a→p) δ_a (k_a·k_v)
//     (and the same with q_v). So the O(D²) work is one dense product per head,
//         P = S_0 · [K | Q]      (M = Dv rows, K = Dk, N = 2T columns),
//     plus the small Gram block k_a·[K|Q] and an O(T²) recurrence per state row for δ and o.
//   * P runs on the 5th-generation tensor cores (tcgen05.mma kind::tf32, fp32 accumulators in
//     TMEM) in three TF32 products for fp32 accuracy: with x = hi + lo, hi = x truncated to TF32
//     (exactly what the tensor core reads from an fp32 word) and lo = x − hi exact in fp32,
//         P ≈ S_hi·X_hi + S_hi·X_lo + S_lo·X_hi.
//     The first two share one pass over the state tile (B = [X_hi ; X_lo], N = 4T); the tile is
//     then overwritten in place by S_lo for the second pass. The tensor core reads its operands
//     from shared memory, so the number of passes over the 64 KiB tile is what it costs.
//   * One 256-thread CTA per (l, b, h). At entry one thread starts the 2-D TMA of the head's S_0
//     tile (row-major, 128-byte-swizzled K-major boxes: directly the UMMA operand layout) and a
//     warp starts 1-D bulk copies of the head's qkv / conv-state / conv-weight / gate rows into
//     shared memory; conv, norms, [K|Q] and the Gram block (CUDA cores) overlap the state load.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gdn {

template <typename IO, int D, int TMAX, bool TREE, bool GDK = false>
struct VerifyCfg {
    static constexpr int NWARP = 8;
    static constexpr int NTHR = 256;
    static constexpr int ES = int(sizeof(IO));
    static constexpr int KB = D / 32;                        // K-blocks of 32 tf32 (128 bytes)
    static constexpr int NP = 2 * TMAX < 16 ? 16 : 2 * TMAX; // columns k_*, q_*, zero padding
    static constexpr int XROWS = 2 * NP;                     // B tile rows: X_hi then X_lo
    static constexpr int XKB = XROWS * 128;                  // bytes per K-block of the B tile
    static constexpr int X_BYTES = KB * XKB;
    static constexpr int A_KB = 128 * 128;                   // bytes per K-block of A (M = 128)
    static constexpr int A_BYTES = KB * A_KB;
    static constexpr int TMEM_COLS = XROWS <= 32 ? 32 : (XROWS <= 64 ? 64 : 128);
    // staging of the head's raw inputs: [3 parts q,k,v][W-1+T rows][D] and conv taps [3][D][W];
    // reused for the plain [K|Q] copy once the conv has read it
    static constexpr int XP_STRIDE = D + 4;                  // floats per plain row (padded)
    static constexpr int XP_BYTES = 2 * TMAX * XP_STRIDE * 4;

    // meta block (floats)
    static constexpr int M_GAM = 0, M_BET = M_GAM + TMAX, M_C0 = M_BET + TMAX,
                         M_KQ = M_C0 + TMAX, M_INV = M_KQ + TMAX, M_NRM = M_INV + 2 * TMAX,
                         M_CK = M_NRM + NWARP * TMAX, M_CQ = M_CK + TMAX * TMAX,
                         M_DL = M_CQ + TMAX * TMAX, M_GA = M_DL + (TREE ? TMAX * D : 0),
                         M_FLOATS = M_GA + (GDK ? TMAX * D : 0);
    static constexpr int I_PAR = 0, I_NANC = I_PAR + TMAX, I_ANC = I_NANC + TMAX,
                         I_WIN = I_ANC + (TREE ? TMAX * TMAX : 0),
                         I_FLAG = I_WIN + (TREE ? TMAX * 4 : 0), I_INTS = I_FLAG + 4;

    static constexpr size_t OFF_X = 0;
    static constexpr size_t OFF_A = OFF_X + X_BYTES;
    static constexpr size_t OFF_MF = OFF_A + A_BYTES;
    static constexpr size_t OFF_MI = OFF_MF + size_t(M_FLOATS) * 4;
    static constexpr size_t OFF_BAR = (OFF_MI + size_t(I_INTS) * 4 + 15) / 16 * 16;
    static constexpr size_t OFF_TSLOT = OFF_BAR + 3 * 8;
    static constexpr size_t OFF_STAGE = (OFF_TSLOT + 16 + 127) / 128 * 128;

    static __host__ __device__ constexpr size_t stage_bytes(int T_, int W_) {
        const size_t raw = size_t(3) * (W_ - 1 + T_) * D * ES + size_t(3) * D * W_ * ES;
        return raw > size_t(XP_BYTES) ? raw : size_t(XP_BYTES);
    }
    static __host__ __device__ constexpr size_t smem_bytes(int T_, int W_) {
        return OFF_STAGE + stage_bytes(T_, W_) + 1024;   // + alignment slack for the base
    }

    static_assert(D == 32 || D == 64 || D == 128, "head dim");
    static_assert(OFF_A % 1024 == 0, "swizzle atoms need 1024-byte bases");
};

__device__ __forceinline__ float tf32_trunc(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// y · sigmoid(y) = y / (1 + 2^(−y·log2 e)) on the special-function unit: ex2.approx and
// rcp.approx, each within a few ulp (relative error ~1e-6 overall); subnormals flush to zero, so
// very negative y gives 2^+big = +inf and a result of −0, very positive y gives y.
__device__ __forceinline__ float silu_fast(float y) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(y * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return y * r;
}

// Sum each of V per-lane values over the warp by recursive halving: V-1 + log2(32/V) shuffles.
// Returns the total of value index *idx (valid in every lane; lanes sharing idx agree).
template <int V>
__device__ __forceinline__ float warp_sum_many(float (&v)[V], int lane, int* idx) {
    int base = 0;
#pragma unroll
    for (int m = V, o = 16; m > 1; m >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < m / 2; ++k) {
            const float send = up ? v[k] : v[k + m / 2];
            const float keep = up ? v[k + m / 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        base += up ? m / 2 : 0;
    }
    float s = v[0];
#pragma unroll
    for (int o = 16 / V; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    *idx = base;
    return s;
}

template <typename IO>
__device__ __forceinline__ float io_to_f(IO x) {
    if constexpr (sizeof(IO) == 2) return __bfloat162float(x);
    else return x;
}

template <typename IO, int D, int TMAX, bool TREE, bool GDK>
__global__ void __launch_bounds__(256)
gdn_verify_kernel(const VerifyArgs a, const __grid_constant__ CUtensorMap smap) {
    using Cfg = VerifyCfg<IO, D, TMAX, TREE, GDK>;
    using Tr = IoTraits<IO>;
    constexpr int NP = Cfg::NP, KB = Cfg::KB, XKB = Cfg::XKB, XS = Cfg::XP_STRIDE;

    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that every access stays
    // a shared-memory access for the compiler
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* Xb = smem + Cfg::OFF_X;          // B tile: [K-block][X_hi rows; X_lo rows]
    unsigned char* As = smem + Cfg::OFF_A;          // S_0 tile (then S_lo)
    float* mf = reinterpret_cast<float*>(smem + Cfg::OFF_MF);
    int* mi = reinterpret_cast<int*>(smem + Cfg::OFF_MI);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);   // TMA, inputs, MMA
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TSLOT);
    unsigned char* stage = smem + Cfg::OFF_STAGE;
    float* gam = mf + Cfg::M_GAM;
    float* bet = mf + Cfg::M_BET;
    float* c0 = mf + Cfg::M_C0;
    float* kqv = mf + Cfg::M_KQ;
    float* inv = mf + Cfg::M_INV;
    float* nrm = mf + Cfg::M_NRM;
    float* CK = mf + Cfg::M_CK;
    float* CQ = mf + Cfg::M_CQ;
    float* DL = mf + Cfg::M_DL;
    float* GA = mf + Cfg::M_GA;                     // per-key-channel gates a_t[j] (GDK)
    int* par = mi + Cfg::I_PAR;
    int* nanc = mi + Cfg::I_NANC;
    int* anc = mi + Cfg::I_ANC;
    int* win = mi + Cfg::I_WIN;
    int* flag = mi + Cfg::I_FLAG;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
    const int T = a.T, Hk = a.Hk, Hv = a.Hv, C = a.C, W = a.W;
    const int group = Hv / Hk, kh = h / group;
    const size_t lb = size_t(l) * a.B + b;
    const int NR = W - 1 + T;                       // staged rows per part

    // staging layout (bytes from `stage`)
    IO* qs = reinterpret_cast<IO*>(stage);                                   // [3][NR][D]
    IO* cws = qs + size_t(3) * NR * D;                                       // [3][D][W]
    float* XP = reinterpret_cast<float*>(stage);    // later: plain [K|Q] rows, stride XS

    // ---- 0. state tile by 2-D TMA; raw input rows by 1-D bulk copies; TMEM
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&bar[0], 1);
            mbar_init(&bar[1], 1);
            mbar_init(&bar[2], 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&bar[0], uint32_t(D) * D * 4);
            const int row0 = int((lb * Hv + h) * D);
            for (int kb = 0; kb < KB; ++kb)
                tma_load_2d(As + kb * Cfg::A_KB, &smap, kb * 32, row0, &bar[0]);
            const uint32_t in_bytes = uint32_t(3 * NR * D * Cfg::ES + 3 * D * W * Cfg::ES);
            mbar_arrive_expect_tx(&bar[1], in_bytes);
            flag[0] = 0;
        }
        __syncwarp();
        const IO* qkv = static_cast<const IO*>(a.qkv);
        const IO* cst = static_cast<const IO*>(a.conv_state);
        const IO* cw = static_cast<const IO*>(a.conv_w);
        const int ncopy = 3 * NR + 3;
        for (int i = lane; i < ncopy; i += 32) {
            const void* src;
            void* dst;
            uint32_t bytes;
            if (i < 3 * NR) {
                const int p = i / NR, r = i - p * NR;
                const int cb = p == 0 ? kh * D : (p == 1 ? Hk * D + kh * D : 2 * Hk * D + h * D);
                src = r < W - 1 ? static_cast<const void*>(cst + (lb * (W - 1) + r) * size_t(C) + cb)
                                : static_cast<const void*>(qkv + (lb * T + (r - (W - 1))) * size_t(C) + cb);
                dst = qs + size_t(i) * D;
                bytes = uint32_t(D * Cfg::ES);
            } else {
                const int p = i - 3 * NR;
                const int cb = p == 0 ? kh * D : (p == 1 ? Hk * D + kh * D : 2 * Hk * D + h * D);
                src = cw + (size_t(l) * C + cb) * W;
                dst = cws + size_t(p) * D * W;
                bytes = uint32_t(D * W * Cfg::ES);
            }
            bulk_g2s(dst, src, bytes, &bar[1]);
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tslot)), "r"(uint32_t(Cfg::TMEM_COLS)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if constexpr (TREE) {
        if (tid < T) par[tid] = __ldg(a.parent + size_t(b) * T + tid);
    }
    // this thread's gate pair (tid < T): loaded now, stored once the conv is under way
    float g_in = 0.f, b_in = 0.f;
    if (tid < T) {
        if constexpr (!GDK) g_in = __ldg(a.g + (lb * T + tid) * Hv + h);
        b_in = __ldg(a.beta + (lb * T + tid) * Hv + h);
    }
    if constexpr (GDK) {   // the head's T x D gate rows, coalesced, into the meta block
        for (int e = tid; e < T * D; e += Cfg::NTHR)
            GA[e] = __ldg(a.g + ((lb * T + e / D) * Hv + h) * size_t(D) + (e % D));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    // ---- 1. tree topology: validate parents, conv windows
    bool skip = false;
    if constexpr (TREE) {
        if (tid < T) {
            const int p = par[tid];
            if (p < -1 || p >= tid) atomicOr(flag, 1);
        }
        __syncthreads();
        skip = flag[0] != 0;
        if (!skip && tid < T) {
            int x = tid, e = 0;
            for (int d = 0; d < 4; ++d) {
                int src = -1;
                if (d < W) {
                    if (x >= 0) { src = (W - 1) + x; x = par[x]; }
                    else { src = (W - 2) - e; ++e; }
                }
                win[tid * 4 + d] = src;
            }
        }
    }
    if (!mbar_wait_bounded(&bar[1], 0) && tid == 0) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
    if (tid < T) {
        gam[tid] = g_in;
        bet[tid] = b_in;
    }
    __syncthreads();
    if (skip) {   // bad tree: report, let the TMA land, free TMEM, leave
        if (tid == 0) {
            set_status(a.status, GDN_STATUS_BAD_PARENT);
            if (!mbar_wait_bounded(&bar[0], 0)) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 1)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                         ::"r"(tbase), "r"(uint32_t(Cfg::TMEM_COLS)));
        return;
    }

    // ---- 2. causal depthwise conv + SiLU from the staged rows. Threads [0, D): q and v channels
    //         of row idx; threads [D, 2D): k channels. (Value row i = thread i keeps its v.)
    const int part = tid / D, idx = tid - part * D;
    float yqk[TMAX], yv[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) { yqk[t] = 0.f; yv[t] = 0.f; }
    if (part < 2) {
#pragma unroll
        for (int pc = 0; pc < 2; ++pc) {
            if (pc == 1 && part == 1) break;
            const int p = part == 1 ? 1 : (pc == 0 ? 0 : 2);
            const IO* col = qs + size_t(p) * NR * D + idx;     // column of channel idx, part p
            const IO* wp = cws + (size_t(p) * D + idx) * W;
            float wr[4];  // wr[d] multiplies the row at distance d (0 = current token)
#pragma unroll
            for (int d = 0; d < 4; ++d) wr[d] = (d < W) ? io_to_f(wp[W - 1 - d]) : 0.f;
            float y[TMAX];
            if constexpr (!TREE) {
                float E[3 + TMAX];
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int r = k + W - 4;
                    E[k] = (r >= 0) ? io_to_f(col[size_t(r) * D]) : 0.f;
                }
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
                    E[3 + t] = (t < T) ? io_to_f(col[size_t(W - 1 + t) * D]) : 0.f;
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    float acc = wr[3] * E[t];
                    acc = fmaf(wr[2], E[t + 1], acc);
                    acc = fmaf(wr[1], E[t + 2], acc);
                    acc = fmaf(wr[0], E[t + 3], acc);
                    y[t] = (t < T) ? silu_fast(acc) : 0.f;
                }
            } else {
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    float acc = 0.f;
                    if (t < T) {
#pragma unroll
                        for (int d = 3; d >= 0; --d) {
                            const int src = win[t * 4 + d];     // staged row index
                            if (src >= 0) acc = fmaf(wr[d], io_to_f(col[size_t(src) * D]), acc);
                        }
                        acc = silu_fast(acc);
                    }
                    y[t] = acc;
                }
            }
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                if (pc == 0) yqk[t] = y[t];
                else yv[t] = y[t];
            }
        }
    }

    // ---- 3. L2 norms of q_t (warps of part 0) and k_t (part 1), per head over D channels
    {
        float sq[TMAX];
#pragma unroll
        for (int t = 0; t < TMAX; ++t) sq[t] = yqk[t] * yqk[t];
        int ix;
        const float s = warp_sum_many<TMAX>(sq, lane, &ix);
        if ((lane & (32 / TMAX - 1)) == 0) nrm[warp * TMAX + ix] = s;
    }
    __syncthreads();   // also: every read of the staged rows is done, XP may overwrite them
    if (tid < 2 * TMAX) {
        // column c < TMAX: k_c (part-1 warps), c >= TMAX: q (part-0 warps)
        const int t = tid < TMAX ? tid : tid - TMAX;
        const int want = tid < TMAX ? 1 : 0;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < Cfg::NWARP; ++w)
            if ((w * 32) / D == want) s += nrm[w * TMAX + t];
        inv[tid] = 1.0f / sqrtf(s + a.l2_eps);
    }
    __syncthreads();
    // [K|Q] columns: n < TMAX -> k_n, TMAX <= n < 2 TMAX -> q, the rest zero. B tile rows n
    // (hi) and NP + n (lo) in the swizzled K-major layout; plain fp32 rows XP[n] for the Gram.
    // Per-key-channel gates: the tile holds A_t ⊙ k_t and A_t ⊙ q_t with A_t[j] = Π_{r≤t} a_r[j]
    // (S_0 decayed to step t, seen through column j); XP and the tape keep the plain vectors.
    if (part < 2) {
        const int n0 = part == 1 ? 0 : TMAX;
        float cum = 1.f;
#pragma unroll
        for (int t = 0; t < TMAX; ++t) {
            const float x = yqk[t] * inv[n0 + t];
            float xw = x;
            if constexpr (GDK) {
                if constexpr (TREE) {          // the gates of t and its ancestors, root-most last
                    cum = 1.f;
                    if (t < T)
                        for (int y = t; y >= 0; y = par[y]) cum *= GA[y * D + idx];
                } else if (t < T) {
                    cum *= GA[t * D + idx];
                }
                xw = x * cum;
            }
            const float hi = tf32_trunc(xw);
            *reinterpret_cast<float*>(Xb + sw128_off(n0 + t, idx, XKB)) = hi;
            *reinterpret_cast<float*>(Xb + sw128_off(NP + n0 + t, idx, XKB)) = xw - hi;
            XP[(n0 + t) * XS + idx] = x;
            if (part == 1 && (h % group) == 0 && t < T)
                a.tape_k[((lb * T + t) * Hk + kh) * size_t(D) + idx] = x;
        }
        if (part == 0) {
#pragma unroll
            for (int n = 2 * TMAX; n < NP; ++n) {
                *reinterpret_cast<float*>(Xb + sw128_off(n, idx, XKB)) = 0.f;
                *reinterpret_cast<float*>(Xb + sw128_off(NP + n, idx, XKB)) = 0.f;
            }
            if constexpr (TREE) {
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
                    if (t < T) DL[size_t(t) * D + idx] = yv[t];
            }
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- 4. tensor cores, first pass over S_0: P[:, 0:NP] = S_hi·X_hi, P[:, NP:2NP] = S_hi·X_lo
    const uint32_t sX = smem_u32(Xb), sA = smem_u32(As);
    if (tid == 0) {
        if (!mbar_wait_bounded(&bar[0], 0)) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
        tc_fence_after();
        constexpr uint32_t IDESC1 = umma_idesc_tf32(128, 2 * NP);
        const uint64_t da = umma_desc_sw128(sA), db = umma_desc_sw128(sX);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_tf32(tbase, da + uint64_t((kb * Cfg::A_KB + ks * 32) >> 4),
                          db + uint64_t((kb * XKB + ks * 32) >> 4), IDESC1, (kb | ks) ? 1u : 0u);
        umma_commit(&bar[2]);
    }
    __syncwarp();

    // ---- 5. Gram block on CUDA cores: G[a][c] = k_a · X_c (a < TMAX, c < 2 TMAX), 2 threads
    //         per entry; CK[v][a] = k_a·k_v, CQ[v][a] = k_a·q_v
    if constexpr (GDK) {
        // Per-key-channel gates: the decay between write s and read t differs per column j, so
        // the Gram carries it, CK[t][s] = Σ_j k_s[j] k_t[j] Π_{s<r≤t} a_r[j] (CQ with q_t), built
        // as a running product per (s, j) in 8-lane groups (thread: s = tid/8, j ≡ tid mod 8),
        // never as a ratio of cumulative products (which underflow). kqv[s] = k_s·q_s.
        constexpr int NJ = D / 8;
        const int s = tid >> 3, c = tid & 7;
        const bool act = s < T;
        float ks[NJ], w[NJ];
        float kq = 0.f;
#pragma unroll
        for (int m = 0; m < NJ; ++m) {
            const int j = c + 8 * m;
            w[m] = 1.f;
            ks[m] = 0.f;
            if (act) {                     // rows s and TMAX + s exist only for s < T
                ks[m] = XP[s * XS + j];
                kq = fmaf(ks[m], XP[(TMAX + s) * XS + j], kq);
            }
        }
        kq += __shfl_xor_sync(0xffffffffu, kq, 1);
        kq += __shfl_xor_sync(0xffffffffu, kq, 2);
        kq += __shfl_xor_sync(0xffffffffu, kq, 4);
        if (c == 0 && act) {
            kqv[s] = kq;
            c0[s] = 1.f;
        }
        if constexpr (TREE) {
            // node v = s reads its ancestors x: CK[v][x] = Σ_j k_x[j] k_v[j] Π_{r ∈ (x, v]} a_r[j],
            // the product running up the parent chain (v's own gate first). The 8 lanes of a
            // group share v, so each group reduces with its own lane mask.
            const unsigned gmask = 0xFFu << (lane & 24);
            const int v = s;
#pragma unroll
            for (int m = 0; m < NJ; ++m) w[m] = act ? GA[v * D + c + 8 * m] : 1.f;
            for (int x = act ? par[v] : -1; x >= 0; x = par[x]) {
                float ck = 0.f, cq = 0.f;
#pragma unroll
                for (int m = 0; m < NJ; ++m) {
                    const int j = c + 8 * m;
                    const float xw = XP[x * XS + j] * w[m];
                    ck = fmaf(xw, ks[m], ck);
                    cq = fmaf(xw, XP[(TMAX + v) * XS + j], cq);
                    w[m] *= GA[x * D + j];
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    ck += __shfl_xor_sync(gmask, ck, o);
                    cq += __shfl_xor_sync(gmask, cq, o);
                }
                if (c == 0) {
                    CK[v * TMAX + x] = ck;
                    CQ[v * TMAX + x] = cq;
                }
            }
        } else
        for (int t = 1; t < T; ++t) {          // warp-uniform trip count (shuffles below)
            const bool on = t > s;
            float ck = 0.f, cq = 0.f;
#pragma unroll
            for (int m = 0; m < NJ; ++m) {
                const int j = c + 8 * m;
                w[m] *= on ? GA[t * D + j] : 1.f;
                const float kw = ks[m] * w[m];
                ck = fmaf(kw, XP[t * XS + j], ck);
                cq = fmaf(kw, XP[(TMAX + t) * XS + j], cq);
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                ck += __shfl_xor_sync(0xffffffffu, ck, o);
                cq += __shfl_xor_sync(0xffffffffu, cq, o);
            }
            if (c == 0 && on) {
                CK[t * TMAX + s] = ck;
                CQ[t * TMAX + s] = cq;
            }
        }
    } else {
        constexpr int NENT = TMAX * 2 * TMAX;
        const int half = tid & 1;
        for (int e = tid >> 1; e < NENT; e += Cfg::NTHR / 2) {
            const int an = e / (2 * TMAX), c = e - an * (2 * TMAX);
            const float4* xa = reinterpret_cast<const float4*>(XP + an * XS + half * (D / 2));
            const float4* xc = reinterpret_cast<const float4*>(XP + c * XS + half * (D / 2));
            float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
            for (int q = 0; q < D / 8; ++q) {
                const float4 u = xa[q], w = xc[q];
                s0 = fmaf(u.x, w.x, s0);
                s1 = fmaf(u.y, w.y, s1);
                s0 = fmaf(u.z, w.z, s0);
                s1 = fmaf(u.w, w.w, s1);
            }
            float s = s0 + s1;
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            if (half == 0) {
                if (c < TMAX) CK[c * TMAX + an] = s;
                else CQ[(c - TMAX) * TMAX + an] = s;
            }
        }
    }
    // fold the gate products in: CK[v][a] *= Γ(a→parent(v)); c0[v] = Γ(root→parent(v)) (the
    // per-channel Gram above already carries its decays, and c0 = 1); trees list each node's
    // ancestors for the recurrence
    if constexpr (!GDK || TREE) {
        __syncthreads();
        if (tid < T) {
            const int v = tid;
            float coef = 1.f;
            int m = 0;
            int x = TREE ? par[v] : v - 1;
            if constexpr (!GDK) kqv[v] = CQ[v * TMAX + v];
            while (x >= 0) {
                if constexpr (!GDK) {
                    CK[v * TMAX + x] *= coef;
                    CQ[v * TMAX + x] *= coef;
                    coef *= gam[x];
                }
                if constexpr (TREE) anc[v * TMAX + m] = x;
                ++m;
                x = TREE ? par[x] : x - 1;
            }
            if constexpr (!GDK) c0[v] = coef;
            if constexpr (TREE) nanc[v] = m;
        }
    }

    // ---- 6. once the first pass is done: S_0 tile -> S_lo in place; second pass S_lo·X_hi
    if (!mbar_wait_bounded(&bar[2], 0) && lane == 0) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
    tc_fence_after();
    {
        constexpr int CHUNKS = KB * D * 8;          // 16-byte chunks of rows < D
#pragma unroll 4
        for (int c = tid; c < CHUNKS; c += Cfg::NTHR) {
            const int kb = c / (D * 8), w = c - kb * (D * 8);
            float4* p = reinterpret_cast<float4*>(As + kb * Cfg::A_KB + w * 16);
            float4 v = *p;
            v.x -= tf32_trunc(v.x);
            v.y -= tf32_trunc(v.y);
            v.z -= tf32_trunc(v.z);
            v.w -= tf32_trunc(v.w);
            *p = v;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        constexpr uint32_t IDESC2 = umma_idesc_tf32(128, NP);
        const uint64_t da = umma_desc_sw128(sA), db = umma_desc_sw128(sX);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_tf32(tbase, da + uint64_t((kb * Cfg::A_KB + ks * 32) >> 4),
                          db + uint64_t((kb * XKB + ks * 32) >> 4), IDESC2, 1u);
        umma_commit(&bar[2]);
    }
    __syncwarp();
    if (!mbar_wait_bounded(&bar[2], 1) && lane == 0) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
    tc_fence_after();

    // ---- 7. per-row recurrence for δ and o (thread = state row i, TMEM lane i)
    if (tid < D) {
        float pr[2 * NP];
#pragma unroll
        for (int c = 0; c < 2 * NP; c += 16) tmem_ld16(tbase + (uint32_t(warp * 32) << 16) + c, pr + c);
#pragma unroll
        for (int c = 0; c < NP; ++c) pr[c] += pr[NP + c];     // + S_hi·X_lo
        const int i = tid;
        IO* out = static_cast<IO*>(a.out);
        const float scale = a.qk_scale;
        if constexpr (!TREE) {
            float dl[TMAX];
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                dl[t] = 0.f;
                if (t < T) {
                    float sk = c0[t] * pr[t], sq = c0[t] * pr[TMAX + t];
#pragma unroll
                    for (int s = 0; s < t; ++s) {
                        sk = fmaf(CK[t * TMAX + s], dl[s], sk);
                        sq = fmaf(CQ[t * TMAX + s], dl[s], sq);
                    }
                    const float gt = GDK ? 1.f : gam[t];   // per-channel decay: in pr and CK
                    const float u = gt * sk;
                    const float d = bet[t] * (yv[t] - u);
                    dl[t] = d;
                    const float o = scale * fmaf(d, kqv[t], gt * sq);
                    const size_t oi = ((lb * T + t) * Hv + h) * size_t(D) + i;
                    a.tape_delta[oi] = d;
                    Tr::store(out, oi, o);
                }
            }
        } else {
#pragma unroll
            for (int v = 0; v < TMAX; ++v) {
                if (v < T) {
                    const float ca = c0[v];
                    float sk = ca * pr[v], sq = ca * pr[TMAX + v];
                    const int m = nanc[v];
#pragma unroll 1
                    for (int q = 0; q < m; ++q) {
                        const int an = anc[v * TMAX + q];
                        const float da = DL[size_t(an) * D + i];
                        sk = fmaf(CK[v * TMAX + an], da, sk);
                        sq = fmaf(CQ[v * TMAX + an], da, sq);
                    }
                    const float gv = GDK ? 1.f : gam[v];   // per-channel decay: in pr and CK
                    const float u = gv * sk;
                    const float d = bet[v] * (DL[size_t(v) * D + i] - u);
                    DL[size_t(v) * D + i] = d;
                    const float o = scale * fmaf(d, kqv[v], gv * sq);
                    const size_t oi = ((lb * T + v) * Hv + h) * size_t(D) + i;
                    a.tape_delta[oi] = d;
                    Tr::store(out, oi, o);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tbase), "r"(uint32_t(Cfg::TMEM_COLS)));
}

template <typename IO, int D, int TMAX, bool TREE, bool GDK>
cudaError_t launch_verify_t(const VerifyArgs& a, const CUtensorMap& map, cudaStream_t stream) {
    using Cfg = VerifyCfg<IO, D, TMAX, TREE, GDK>;
    auto kern = gdn_verify_kernel<IO, D, TMAX, TREE, GDK>;
    const size_t smem = Cfg::smem_bytes(a.T, a.W);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    const cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hv, a.B, a.L);
    kern<<<grid, Cfg::NTHR, smem, stream>>>(a, map);
    return cudaGetLastError();
}

template <typename IO, bool TREE, bool GDK>
cudaError_t launch_verify_gk(const VerifyArgs& a, const CUtensorMap& map, int D, cudaStream_t s) {
    const int tm = a.T <= 4 ? 4 : a.T <= 8 ? 8 : a.T <= 16 ? 16 : 32;
#define GDN_V_CASE(DD, TM) \
    if (D == DD && tm == TM) return launch_verify_t<IO, DD, TM, TREE, GDK>(a, map, s);
    GDN_V_CASE(32, 4) GDN_V_CASE(32, 8) GDN_V_CASE(32, 16) GDN_V_CASE(32, 32)
    GDN_V_CASE(64, 4) GDN_V_CASE(64, 8) GDN_V_CASE(64, 16) GDN_V_CASE(64, 32)
    GDN_V_CASE(128, 4) GDN_V_CASE(128, 8) GDN_V_CASE(128, 16) GDN_V_CASE(128, 32)
#undef GDN_V_CASE
    return cudaErrorInvalidValue;
}

template <typename IO, bool TREE>
cudaError_t launch_verify_io(const VerifyArgs& a, const CUtensorMap& map, int D, cudaStream_t s) {
    if constexpr (TREE) {
        return a.gate_dk ? launch_verify_gk<IO, true, true>(a, map, D, s)
                         : launch_verify_gk<IO, true, false>(a, map, D, s);
    } else {
        return a.gate_dk ? launch_verify_gk<IO, false, true>(a, map, D, s)
                         : launch_verify_gk<IO, false, false>(a, map, D, s);
    }
}

}  // namespace gdn
