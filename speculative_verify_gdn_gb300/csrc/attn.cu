// attn.cu — the hybrid's full-attention layers in the verify step: append the T verify positions'
// key / value rows to the KV cache, causal GQA attention of those positions over the cache, and
// the KV truncation on reject (sm_103a, tcgen05 tensor cores).
//
// "Speculative Decoding on GDN Hybrid Architectures: A 31-Experiment Investigation", §2.1 (the
// hybrid's attention layers are standard multi-head attention over a KV cache) and §2.2 (their
// N verify positions run in one parallel pass, unlike the GDN layers).
//
// GB300 design:
//   * A small kernel appends the T new rows; the attention kernel then reads every key through
//     TMA. The K cache is token-major [ctx][D]; the V cache is stored transposed per 128-key tile,
//     [ctx/128][D][128], so both tensor-core products read K-major, 128-byte-swizzled tiles exactly
//     as the TMA boxes land and every tile of K and of V is one contiguous 64 KiB block in HBM (a
//     plain [D][ctx] transpose reads 256-byte pieces 2·ctx bytes apart and ran ~5 % slower).
//   * Up to 64 query rows per kv head: one CTA per (layer, sequence, kv head, key split). Its
//     query rows are T·(Hq/Hkv) (position, head) pairs of the kv head, zero-padded to NQ ∈ {32,
//     64}. (65 to 128 rows run in the kernel further below, with the rows on the TMEM lanes.) Per
//     128-key tile:
//         Sᵀ[key][row]  = K_tile · Qᵀ       tcgen05, M = 128 keys, N = NQ, K = D
//         Oᵀ[d][row]   += Vᵀ_tile · Pᵀ      tcgen05, M = 128 d-rows per chunk, N = NQ, K = 128 keys
//     Sᵀ is double-buffered in TMEM (the next tile's product overlaps this tile's softmax) and
//     Oᵀ accumulates in TMEM across the tiles.
//   * Softmax: one warp per (TMEM lane quarter, 32 query columns), thread = key = TMEM lane. The
//     running maximum of a column moves only when a tile holds a score more than 8 (log2 units)
//     above it, so in the common case a tile costs each thread one compare per score and one
//     barrier; otherwise the tile maxima are reduced (a transposing warp reduction, 31 shuffles per
//     32 columns, plus a 4-way shared-memory step) and Oᵀ and the partial sums are rescaled. The
//     weights stay ≤ 2^8; P is rounded to bf16 for the tensor core (one buffer: the softmax is
//     not on the critical path, the shared memory is worth more as a ring stage) and each thread
//     sums its rounded weights, reduced once at the end, so numerator and denominator use the
//     same weights.
//   * Warp roles: softmax + epilogue, then one TMA producer warp, then one MMA issue + TMEM owner
//     warp. The ring holds 32 KiB chunks (128 keys × 128 of the head dim, or 128 d-rows × 128
//     keys), as many as the shared memory left over holds, in the order the tensor core consumes
//     them: K(0), K(1), V(0), K(2), V(1), … Each CTA is bound by the bytes it keeps in flight, so
//     shared memory goes to ring stages first.
//   * Short batches over long caches split the keys across CTAs (flash-decoding); a combine
//     kernel merges the partial (max, sum, O).
// Every wait is bounded (1 s); a timeout sets GDN_STATUS_WAIT_TIMEOUT, the CTA stops issuing
// work, lets its copies land, waits for its tensor-core work and frees its TMEM.
#include "common.cuh"
#include "kernels.h"
#include "attn.h"
#include "tc.cuh"

namespace gdn {

template <int D, int NQ>
struct AttnCfg {
    // softmax warps: one per (TMEM lane quarter, 32 query columns), so every SM sub-partition
    // interleaves NQ / 32 of them
    static constexpr int NSW = 4 * (NQ / 32);
    static constexpr int SMT = 32 * NSW;                // softmax threads
    static constexpr int CW = 32;                       // columns per softmax warp
    static constexpr int PRODUCER = NSW, MMAW = NSW + 1;
    static constexpr int NTHR = 32 * (NSW + 2);
    static constexpr int DCH = D / 128;                 // 128-wide chunks of the head dim
    static constexpr int CHUNK = 128 * 128 * 2;         // one ring stage: two 64-wide swizzled blocks
    static constexpr int Q_KB = NQ * 128;               // bytes of one 64-element K-block of Q
    static constexpr int Q_BYTES = (D / 64) * Q_KB;
    static constexpr int P_KB = NQ * 128;               // bytes of one 64-key K-block of P
    static constexpr int P_BYTES = 2 * P_KB;            // the P tile (one buffer: its smem is
                                                        // worth more as a ring stage)
    // ring stages: as many as the shared memory left over holds (at most 6)
    static constexpr int FIXED = Q_BYTES + P_BYTES + 12 * NQ * 4 + 21 * 8 + 16 + 1024 + 64;
    static constexpr int NST_FIT = (227 * 1024 - FIXED) / CHUNK;
    static constexpr int NST = NST_FIT > 6 ? 6 : NST_FIT;
    static constexpr size_t OFF_RING = 0;
    static constexpr size_t OFF_Q = OFF_RING + size_t(NST) * CHUNK;
    static constexpr size_t OFF_P = OFF_Q + Q_BYTES;
    static constexpr size_t OFF_F = OFF_P + P_BYTES;    // redA[4][NQ] redB[4][NQ] m, alpha, l [NQ]
    static constexpr size_t OFF_LIM = OFF_F + size_t(11) * NQ * 4;   // int lim[NQ]
    // barriers: full[NST] empty[NST] s_full[2] s_free[2] p_full[2] pv_done[2] fin (one barrier per
    // buffer, so no waiter is ever two phases behind)
    static constexpr int NBAR = 2 * NST + 9;
    static constexpr size_t OFF_BAR = (OFF_LIM + size_t(NQ) * 4 + 7) / 8 * 8;
    static constexpr size_t OFF_MISC = OFF_BAR + size_t(NBAR) * 8;   // abort flag, TMEM slot
    static constexpr size_t SMEM = OFF_MISC + 16 + 1024;             // + base alignment slack
    static constexpr int TM_S = 0;                       // Sᵀ buffers: columns [0, 2 NQ)
    static constexpr int TM_O = 2 * NQ;                  // Oᵀ: DCH blocks of NQ columns
    static constexpr int TM_USED = 2 * NQ + DCH * NQ;
    static constexpr int TM_COLS = TM_USED <= 32 ? 32 : TM_USED <= 64 ? 64 : TM_USED <= 128 ? 128
                                 : TM_USED <= 256 ? 256 : 512;
    static_assert(D == 128 || D == 256, "head dim");
    static_assert(NQ == 32 || NQ == 64 || NQ == 128, "query rows");
    static_assert(TM_USED <= 512, "TMEM columns");
    static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0 && Q_KB % 1024 == 0, "swizzle atoms");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(NST >= 2, "ring stages");
};

// tmem_ld32 without the wait: the caller issues tmem_wait_ld() before reading v (several loads
// may then share one wait)
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] · B[smem descriptor]ᵀ, kind::f16 with bf16 operands (A: rows on the TMEM
// lanes, two K elements per 32-bit column, the lower one in the low half). Whole warp, one
// elected lane issues.
__device__ __forceinline__ void umma_bf16_ts_warp(uint32_t dtmem, uint32_t atmem, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(dtmem), "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Reduce V ≤ 32 per-lane values over the warp, column by column: recursive halving (V - 1
// shuffles) leaves each group of 32 / V lanes with one column, and log2(32 / V) more shuffles
// combine the group. Returns the total of column *col (max or sum); lanes of a group agree.
template <int V, bool MAX>
__device__ __forceinline__ float warp_cols(const float* v0, int lane, int* col) {
    float v[V];
#pragma unroll
    for (int k = 0; k < V; ++k) v[k] = v0[k];
    int base = 0;
#pragma unroll
    for (int m = V, o = 16; m > 1; m >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < m / 2; ++k) {
            const float send = up ? v[k] : v[k + m / 2];
            const float keep = up ? v[k + m / 2] : v[k];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            v[k] = MAX ? fmaxf(keep, got) : keep + got;
        }
        base += up ? m / 2 : 0;
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 / V; o > 0; o >>= 1) {
        const float got = __shfl_xor_sync(0xffffffffu, r, o);
        r = MAX ? fmaxf(r, got) : r + got;
    }
    *col = base;
    return r;
}

// ------------------------------------------------------------------ append the new rows
// One block per (sequence, layer, kv head). Keys: 16-byte pieces of whole rows. Values: position
// p = n0 + i is column p % 128 of row d of tile p / 128, so the new rows go through shared memory
// (16-byte loads, rows padded by two elements against bank conflicts) and consecutive threads
// write consecutive positions of one d-row (contiguous runs in the transposed cache).
__global__ void __launch_bounds__(256) attn_append_kernel(const AttnArgs a) {
    const int b = blockIdx.x, l = blockIdx.y, h = blockIdx.z;
    const int n0 = __ldg(a.kv_len + b);
    if (n0 < 0 || n0 > a.ctx - a.T) {
        if (l == 0 && h == 0 && threadIdx.x == 0) set_status(a.status, GDN_STATUS_BAD_LEN);
        return;
    }
    const size_t lb = size_t(l) * a.B + b;
    const int D = a.D, T = a.T, H = a.Hkv, D8 = a.D / 8;
    if (D > 256) return;                                   // the launcher serves D <= 256
#pragma unroll 4
    for (int e = threadIdx.x; e < T * D8; e += blockDim.x) {
        const int d8 = e % D8, i = e / D8;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.k_new + ((lb * T + i) * H + h) * size_t(D)) + d8);
        reinterpret_cast<uint4*>(a.k_cache + ((lb * H + h) * size_t(a.ctx) + n0 + i) * size_t(D))[d8] = v;
    }
    __shared__ __nv_bfloat16 sv[16384];
    const int NT = a.ctx >> 7, SP = D + 2;
    const int TC = min(T, 16384 / SP);                     // positions per chunk (>= 63)
    const __nv_bfloat16* vsrc = a.v_new + (lb * T * H + h) * size_t(D);
    __nv_bfloat16* vdst = a.vt_cache + (lb * H + h) * size_t(NT) * D * 128;
    for (int i0 = 0; i0 < T; i0 += TC) {
        const int tc = min(TC, T - i0);
        __syncthreads();
#pragma unroll 4
        for (int e = threadIdx.x; e < tc * D8; e += blockDim.x) {
            const int t = e / D8, d8 = e - t * D8;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(vsrc + size_t(i0 + t) * H * D) + d8);
            const __nv_bfloat16* pv = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
            for (int k = 0; k < 8; ++k) sv[t * SP + 8 * d8 + k] = pv[k];
        }
        __syncthreads();
#pragma unroll 4
        for (int e = threadIdx.x; e < tc * D; e += blockDim.x) {
            const int d = e / tc, t = e - d * tc;
            const int p = n0 + i0 + t;
            vdst[((p >> 7) * size_t(D) + d) * 128 + (p & 127)] = sv[t * SP + d];
        }
    }
}

// ------------------------------------------------------------------ attention
// The work of block blk: units 0 .. n_full-1 whole (one block each, writing out), then each of the
// remaining (tail) units as `splits` key ranges whose partial (max, sum, O) the combine kernel
// merges. The tail fills the last wave of CTAs with short blocks instead of a few long ones.
struct AttnWork {
    int unit, split, tail, t0, tmax;
    bool whole;
};
__device__ __forceinline__ AttnWork attn_work(const AttnArgs& a, int blk) {
    AttnWork w;
    if (blk < a.n_full) {
        w.unit = blk; w.split = 0; w.tail = 0; w.t0 = 0; w.tmax = 0x3fffffff; w.whole = true;
    } else {
        const int j = blk - a.n_full;
        w.tail = j / a.splits;
        w.split = j - w.tail * a.splits;
        w.unit = a.n_full + w.tail;
        w.t0 = w.split * a.tiles_per_split;
        w.tmax = a.tiles_per_split;
        w.whole = a.splits == 1;
    }
    return w;
}
// first row of a tail block's partial results in the workspace
__device__ __forceinline__ size_t attn_ws_row(const AttnArgs& a, const AttnWork& w) {
    return (size_t(w.split) * (a.units - a.n_full) + w.tail) * a.nq;
}

// TMA producer of both attention kernels (one lane): the ring in the order the tensor core
// consumes it, K(0), K(1), V(0), K(2), V(1), ..., each stage a 32 KiB chunk of 128 keys x 128 of
// the head dim (K) or 128 d-rows x 128 keys (Vᵀ), as two 64-wide swizzled boxes. Every copy
// issued lands before it returns.
template <int NST, int DCH>
__device__ __forceinline__ void attn_produce(const AttnArgs& a, const CUtensorMap* kmap,
                                             const CUtensorMap* vmap, unsigned char* ring,
                                             uint64_t* full, uint64_t* empty,
                                             volatile int* abort_flag, int lb, int kvh, int t0,
                                             int ntiles) {
    constexpr int D = DCH * 128, CHUNK = 128 * 128 * 2;
    const int krow0 = (lb * a.Hkv + kvh) * a.ctx;                  // K map row of key 0
    const int vrow0 = (lb * a.Hkv + kvh) * (a.ctx >> 7) * D;       // Vᵀ map row of tile 0
    int stage = 0, issued = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto load = [&](bool isv, int tile, int c) {
        if (!ok) return;
        if (!pwait(&empty[stage], ph ^ 1u, abort_flag, a.status)) {
            ok = false;
            return;
        }
        mbar_arrive_expect_tx(&full[stage], uint32_t(CHUNK));
        unsigned char* dst = ring + stage * CHUNK;
        const int key0 = (t0 + tile) * 128;
        if (!isv) {
            tma_load_2d(dst, kmap, c * 128, krow0 + key0, &full[stage]);
            tma_load_2d(dst + 16384, kmap, c * 128 + 64, krow0 + key0, &full[stage]);
        } else {
            const int vrow = vrow0 + (t0 + tile) * D + c * 128;
            tma_load_2d(dst, vmap, 0, vrow, &full[stage]);
            tma_load_2d(dst + 16384, vmap, 64, vrow, &full[stage]);
        }
        ++issued;
        if (++stage == NST) {
            stage = 0;
            ph ^= 1u;
        }
    };
    for (int c = 0; c < DCH; ++c) load(false, 0, c);
    for (int j = 0; j < ntiles; ++j) {
        if (j + 1 < ntiles)
            for (int c = 0; c < DCH; ++c) load(false, j + 1, c);
        for (int c = 0; c < DCH; ++c) load(true, j, c);
    }
    for (int s = 0; s < NST && s < issued; ++s) {
        const int fills = (issued - s + NST - 1) / NST;
        if (!mbar_wait_bounded(&full[s], uint32_t(fills - 1) & 1u))
            set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
    }
}

template <int D, int NQ>
__global__ void __launch_bounds__(AttnCfg<D, NQ>::NTHR, 1)
attn_verify_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
    using Cfg = AttnCfg<D, NQ>;
    constexpr int NST = Cfg::NST, DCH = Cfg::DCH, SMT = Cfg::SMT;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* ring = smem + Cfg::OFF_RING;
    unsigned char* Qs = smem + Cfg::OFF_Q;
    unsigned char* Ps = smem + Cfg::OFF_P;
    float* redA = reinterpret_cast<float*>(smem + Cfg::OFF_F);   // [4][NQ] tile maxima per warp
    float* redB = redA + 4 * NQ;                                  // [4][NQ] tile sums per warp
    float* m_run = redB + 4 * NQ;                                 // running maximum (log2 units)
    float* alpha = m_run + NQ;                                    // this tile's rescale factor
    float* lfin = alpha + NQ;                                     // final normaliser
    int* lim = reinterpret_cast<int*>(smem + Cfg::OFF_LIM);       // last key each row may see
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + NST;
    uint64_t* s_full = empty + NST;
    uint64_t* s_free = s_full + 2;
    uint64_t* p_full = s_free + 2;
    uint64_t* pv_done = p_full + 2;
    uint64_t* fin = pv_done + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnWork wk = attn_work(a, blockIdx.x);
    const int unit = wk.unit;
    constexpr int row0 = 0;                                // first query row of this CTA
    const int kvh = unit % a.Hkv, lb = unit / a.Hkv, b = lb % a.B;
    const int T = a.T, G = a.group;
    const int n0 = __ldg(a.kv_len + b);
    if (n0 < 0 || n0 > a.ctx - T) return;                 // reported by the append kernel
    const int t0 = wk.t0;                                  // first 128-key tile of this CTA
    const int ntiles = min(((n0 + T + 127) >> 7) - t0, wk.tmax);
    if (ntiles <= 0) {                                     // a split past the end: empty partial
        if (tid < NQ && row0 + tid < a.nq) {
            float* ml = a.ws_ml + (attn_ws_row(a, wk) + row0 + tid) * 2;
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&s_free[0], SMT);
        mbar_init(&s_free[1], SMT);
        mbar_init(&p_full[0], SMT);
        mbar_init(&p_full[1], SMT);
        mbar_init(&pv_done[0], 1);
        mbar_init(&pv_done[1], 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == Cfg::MMAW) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tslot)), "r"(uint32_t(Cfg::TM_COLS)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // query rows c = i·G + g (position i, head kvh·G + g) into the K-major swizzled B tile
    {
        const __nv_bfloat16* qh = a.q + (size_t(lb) * T * a.Hq + size_t(kvh) * G) * D;
        for (int e = tid; e < NQ * (D / 8); e += Cfg::NTHR) {
            const int c = e / (D / 8), j8 = e - c * (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row0 + c < a.nq) {
                const int i = (row0 + c) / G, g = (row0 + c) - i * G;
                v = __ldg(reinterpret_cast<const uint4*>(qh + (size_t(i) * a.Hq + g) * D) + j8);
            }
            const int kb = j8 >> 3, ch = j8 & 7;
            *reinterpret_cast<uint4*>(Qs + kb * Cfg::Q_KB + (c >> 3) * 1024 + (c & 7) * 128 +
                                      ((ch ^ (c & 7)) << 4)) = v;
        }
        if (tid < NQ) {
            m_run[tid] = -INFINITY;
            lim[tid] = n0 + (row0 + tid < a.nq ? (row0 + tid) / G : T - 1);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == Cfg::PRODUCER) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0)
            attn_produce<NST, DCH>(a, &kmap, &vmap, ring, full, empty, abort_flag, lb, kvh, t0, ntiles);
        __syncwarp();
    } else if (warp == Cfg::MMAW) {
        // ---------------------------------------------------------------- MMA issue
        constexpr uint32_t IDESC = umma_idesc_bf16(128, NQ);
        const uint32_t sQ = smem_u32(Qs), sP = smem_u32(Ps), sR = smem_u32(ring);
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        auto qk = [&](int j) {
            const int buf = j & 1;
            if (j >= 2 && !pwait_warp(&s_free[buf], uint32_t((j >> 1) - 1) & 1u, abort_flag, a.status)) {
                ok = false;
                return;
            }
            tc_fence_after();
            for (int c = 0; c < DCH; ++c) {
                if (!pwait_warp(&full[stage], ph, abort_flag, a.status)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint64_t da = umma_desc_sw128(sR + stage * Cfg::CHUNK);
                const uint64_t db = umma_desc_sw128(sQ + 2 * c * Cfg::Q_KB);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16_warp(tbase + Cfg::TM_S + buf * NQ,
                                       da + uint64_t((kb * 16384 + ks * 32) >> 4),
                                       db + uint64_t((kb * Cfg::Q_KB + ks * 32) >> 4), IDESC,
                                       (c | kb | ks) ? 1u : 0u);
                umma_commit_warp(&empty[stage]);
                if (++stage == NST) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            umma_commit_warp(&s_full[buf]);
        };
        auto pv = [&](int j) {
            const int buf = j & 1;
            if (!pwait_warp(&p_full[buf], uint32_t(j >> 1) & 1u, abort_flag, a.status)) {
                ok = false;
                return;
            }
            tc_fence_after();
            for (int c = 0; c < DCH; ++c) {
                if (!pwait_warp(&full[stage], ph, abort_flag, a.status)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint64_t da = umma_desc_sw128(sR + stage * Cfg::CHUNK);
                const uint64_t db = umma_desc_sw128(sP);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16_warp(tbase + Cfg::TM_O + c * NQ,
                                       da + uint64_t((kb * 16384 + ks * 32) >> 4),
                                       db + uint64_t((kb * Cfg::P_KB + ks * 32) >> 4), IDESC,
                                       (j > 0 || kb || ks) ? 1u : 0u);
                umma_commit_warp(&empty[stage]);
                if (++stage == NST) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            umma_commit_warp(&pv_done[buf]);
        };
        qk(0);
        for (int j = 0; j < ntiles && ok; ++j) {
            if (j + 1 < ntiles) qk(j + 1);
            if (ok) pv(j);
        }
        umma_commit_warp(fin);          // arrives once every MMA issued above has completed
    } else {
        // ---------------------------------------------------------------- softmax warps
        // warp = (32 query columns from col0, TMEM lane quarter q4); row = key of the tile and
        // d-row of Oᵀ. Per tile the common case is one barrier: each thread checks its scores
        // against the running maxima + 8; only if some score is above (or a wait failed) do the
        // warps reduce the tile maxima, move the maxima and rescale Oᵀ and the partial sums.
        const int q4 = warp & 3, col0 = (warp >> 2) * 32, row = q4 * 32 + lane;
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        const float sl2 = a.sl2;
        float lsum[32];                 // partial normaliser of column col0 + k over this key lane
#pragma unroll
        for (int k = 0; k < 32; ++k) lsum[k] = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int buf = j & 1;
            const int key = (t0 + j) * 128 + row;
            const bool edge = (t0 + j) * 128 + 127 > n0;   // some row cannot see some key here
            ok = pwait(&s_full[buf], uint32_t(j >> 1) & 1u, abort_flag, a.status) && ok;
            tc_fence_after();
            const uint32_t tS = tbase + lane_off + Cfg::TM_S + buf * NQ + col0;
            uint32_t vis = 0xffffffffu;         // bit k: column col0 + k may see this key
            if (edge) {
#pragma unroll
                for (int k = 0; k < 32; ++k) vis &= ~(uint32_t(key > lim[col0 + k]) << k);
            }
            float s[32];
            tmem_ld32(tS, s);
            bool over = false;
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
                const float4 m4 = *reinterpret_cast<const float4*>(m_run + col0 + 4 * k4);
                const float mk[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = 4 * k4 + u;
                    s[k] *= sl2;
                    over |= ((vis >> k) & 1u) && s[k] > mk[u] + 8.f;
                }
            }
            if (named_bar_or(1, SMT, over || !ok)) {
                // slow path: tile maxima of every column, new running maxima, rescale
#pragma unroll
                for (int k = 0; k < 32; ++k) s[k] = ((vis >> k) & 1u) ? s[k] : -INFINITY;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int col;
                    const float mx = warp_cols<16, true>(s + 16 * h, lane, &col);
                    redA[q4 * NQ + col0 + 16 * h + col] = mx;
                }
                named_bar(1, SMT);
                bool resc = false;
                if (tid < NQ) {
                    const float mt = fmaxf(fmaxf(redA[tid], redA[NQ + tid]),
                                           fmaxf(redA[2 * NQ + tid], redA[3 * NQ + tid]));
                    const float mo = m_run[tid];
                    float al = 1.f;
                    if (mt > mo + 8.f) {        // never for mt = -inf (nothing visible yet)
                        al = (mo == -INFINITY) ? 0.f : ex2(mo - mt);
                        m_run[tid] = mt;
                        resc = true;
                    }
                    alpha[tid] = al;
                }
                if (named_bar_or(1, SMT, resc)) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) lsum[k] *= alpha[col0 + k];
                    if (j > 0) {
                        // Oᵀ holds P·V up to tile j-1: that product must be done first
                        ok = pwait(&pv_done[(j - 1) & 1], uint32_t((j - 1) >> 1) & 1u, abort_flag,
                                   a.status) && ok;
                        tc_fence_after();
#pragma unroll 1
                        for (int c2 = 0; c2 < DCH; ++c2) {
                            const uint32_t tO = tbase + lane_off + Cfg::TM_O + c2 * NQ + col0;
                            float o[32];
                            tmem_ld32(tO, o);
#pragma unroll
                            for (int k = 0; k < 32; ++k) o[k] *= alpha[col0 + k];
                            tmem_st32(tO, o);
                        }
                        tmem_wait_st();
                    }
                }
                // the scores again (not kept in registers across the reduction)
                tmem_ld32(tS, s);
#pragma unroll
                for (int k = 0; k < 32; ++k) s[k] *= sl2;
            }
            tc_fence_before();
            mbar_arrive(&s_free[buf]);          // Sᵀ(j) lives in registers now
            // the P tile was last read by P·V of tile j-1
            if (j >= 1)
                ok = pwait(&pv_done[(j - 1) & 1], uint32_t((j - 1) >> 1) & 1u, abort_flag,
                           a.status) && ok;
            unsigned char* Pb = Ps + (row >> 6) * Cfg::P_KB;
            const int rsw = (row & 63) >> 3, rb = (row & 7) * 2;
#pragma unroll
            for (int k4 = 0; k4 < 8; ++k4) {
                const float4 m4 = *reinterpret_cast<const float4*>(m_run + col0 + 4 * k4);
                const float mk[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = 4 * k4 + u, c = col0 + k;
                    float e = ex2(s[k] - mk[u]);
                    e = ((vis >> k) & 1u) ? e : 0.f;
                    const __nv_bfloat16 pb = __float2bfloat16_rn(e);
                    lsum[k] += __bfloat162float(pb);
                    *reinterpret_cast<__nv_bfloat16*>(Pb + (c >> 3) * 1024 + (c & 7) * 128 +
                                                      ((rsw ^ (c & 7)) << 4) + rb) = pb;
                }
            }
            fence_async_smem();                 // P visible to the tensor core
            mbar_arrive(&p_full[buf]);
        }
        // ---------------------------------------------------------------- epilogue
        {   // normalisers: partial sums over the key lanes, then over the lane quarters
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int col;
                const float sm = warp_cols<16, false>(lsum + 16 * h, lane, &col);
                redB[q4 * NQ + col0 + 16 * h + col] = sm;
            }
        }
        ok = pwait(&pv_done[(ntiles - 1) & 1], uint32_t((ntiles - 1) >> 1) & 1u, abort_flag,
                   a.status) && ok;
        named_bar(1, SMT);
        float l_fin = 0.f;
        if (tid < NQ) {
            l_fin = (redB[tid] + redB[NQ + tid]) + (redB[2 * NQ + tid] + redB[3 * NQ + tid]);
            lfin[tid] = l_fin;
        }
        const bool bad = named_bar_or(1, SMT, !ok);
        tc_fence_after();
        if (!bad) {
            const size_t ws_row = attn_ws_row(a, wk);
#pragma unroll 1
            for (int c2 = 0; c2 < DCH; ++c2) {
                float o[32];
                tmem_ld32(tbase + lane_off + Cfg::TM_O + c2 * NQ + col0, o);
                const int d = c2 * 128 + row;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int c = col0 + k, cg = row0 + c;      // local and unit-wide row
                    if (cg < a.nq) {
                        if (wk.whole) {
                            const int i = cg / G, g = cg - i * G;
                            a.out[((size_t(lb) * T + i) * a.Hq + kvh * G + g) * D + d] =
                                __float2bfloat16_rn(o[k] / lfin[c]);
                        } else {
                            a.ws_o[(ws_row + cg) * D + d] = o[k];
                        }
                    }
                }
            }
            if (!wk.whole && tid < NQ && row0 + tid < a.nq) {
                float* ml = a.ws_ml + (ws_row + row0 + tid) * 2;
                ml[0] = m_run[tid];
                ml[1] = l_fin;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::MMAW) {
        tc_fence_after();
        if (!mbar_wait_bounded(fin, 0)) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tbase), "r"(uint32_t(Cfg::TM_COLS)));
    }
}

// ------------------------------------------------------------------ attention, 65-128 query rows
// One CTA per (unit, key split) holds all of a kv head's query rows, on the TMEM lanes (M = 128).
// Per 128-key tile:
//     S[row][key]  = Q · K_tileᵀ     tcgen05, A = Q (shared memory), B = K tile, N = 128 keys
//     O[row][d]   += P · V_tile      tcgen05, A = P (TMEM), B = Vᵀ tile, N = 128 d-rows per chunk
// Two softmax threads per row (TMEM lane), one per half of the tile's keys; the row keeps one
// running maximum, which both threads hold (when a tile may move it, they exchange their tile
// maxima through shared memory).
// P is written back as packed bf16 pairs over the first 64 columns of its tile's S buffer (S is
// double-buffered; tile j+2's scores reuse tile j's buffer once P·V of tile j is done), so the
// shared memory holds only Q (128 rows) and the ring. Each CTA reads every K / V tile of its key
// range once: the 64-row kernel would run these rows as two CTAs, each reading all of them. The
// lazy running maximum, the bf16 weights and the sums of the rounded weights are those of the
// 64-row kernel.
template <int D>
struct AttnRowsCfg {
    static constexpr int NQ = 128, DCH = D / 128;
    // warps 0-7: softmax, warp w on TMEM lane quarter w & 3 and key half w >> 2
    static constexpr int NSW = 8, PRODUCER = 8, MMAW = 9, NTHR = 320;
    static constexpr int CHUNK = 128 * 128 * 2;
    static constexpr int Q_KB = NQ * 128, Q_BYTES = (D / 64) * Q_KB;
    static constexpr int FIXED = Q_BYTES + 2 * NQ * 4 + 17 * 8 + 16 + 1024;
    static constexpr int NST_FIT = (227 * 1024 - FIXED) / CHUNK;
    static constexpr int NST = NST_FIT > 6 ? 6 : NST_FIT;
    static constexpr size_t OFF_RING = 0;
    static constexpr size_t OFF_Q = OFF_RING + size_t(NST) * CHUNK;
    static constexpr size_t OFF_X = OFF_Q + Q_BYTES;               // float xch[2][NQ]
    // barriers: full[NST] empty[NST] s_full[2] p_full[2] pv_done[2] fin
    static constexpr int NBAR = 2 * NST + 7;
    static constexpr size_t OFF_BAR = (OFF_X + size_t(2 * NQ) * 4 + 7) / 8 * 8;
    static constexpr size_t OFF_MISC = OFF_BAR + size_t(NBAR) * 8;   // abort flag, TMEM slot
    static constexpr size_t SMEM = OFF_MISC + 16 + 1024;             // + base alignment slack
    // TMEM: S buffers at [0, 128) and [128, 256) (P over the first 64 columns of each), O at
    // [256, 256 + D)
    static constexpr int TM_S = 0, TM_O = 256, TM_COLS = 512;
    static_assert(D == 128 || D == 256, "head dim");
    static_assert(OFF_Q % 1024 == 0 && Q_KB % 1024 == 0, "swizzle atoms");
    static_assert(SMEM <= 227 * 1024 && NST >= 2, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(AttnRowsCfg<D>::NTHR, 1)
attn_rows_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    using Cfg = AttnRowsCfg<D>;
    constexpr int NST = Cfg::NST, DCH = Cfg::DCH, NQ = Cfg::NQ;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* ring = smem + Cfg::OFF_RING;
    unsigned char* Qs = smem + Cfg::OFF_Q;
    float* xch = reinterpret_cast<float*>(smem + Cfg::OFF_X);      // [key half][row]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + NST;
    uint64_t* s_full = empty + NST;
    uint64_t* p_full = s_full + 2;
    uint64_t* pv_done = p_full + 2;
    uint64_t* fin = pv_done + 2;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const AttnWork wk = attn_work(a, blockIdx.x);
    const int unit = wk.unit;
    const int kvh = unit % a.Hkv, lb = unit / a.Hkv, b = lb % a.B;
    const int T = a.T, G = a.group;
    const int n0 = __ldg(a.kv_len + b);
    if (n0 < 0 || n0 > a.ctx - T) return;                 // reported by the append kernel
    const int t0 = wk.t0;                                  // first 128-key tile of this CTA
    const int ntiles = min(((n0 + T + 127) >> 7) - t0, wk.tmax);
    if (ntiles <= 0) {                                     // a split past the end: empty partial
        if (tid < a.nq) {
            float* ml = a.ws_ml + (attn_ws_row(a, wk) + tid) * 2;
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&s_full[k], 1);
            mbar_init(&p_full[k], Cfg::NSW);           // one lane of each softmax warp
            mbar_init(&pv_done[k], 1);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == Cfg::MMAW) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tslot)), "r"(uint32_t(Cfg::TM_COLS)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // query rows c = i·G + g (position i, head kvh·G + g) into the K-major swizzled A tile, zero
    // beyond nq
    {
        const __nv_bfloat16* qh = a.q + (size_t(lb) * T * a.Hq + size_t(kvh) * G) * D;
        for (int e = tid; e < NQ * (D / 8); e += Cfg::NTHR) {
            const int c = e / (D / 8), j8 = e - c * (D / 8);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (c < a.nq) {
                const int i = c / G, g = c - i * G;
                v = __ldg(reinterpret_cast<const uint4*>(qh + (size_t(i) * a.Hq + g) * D) + j8);
            }
            const int kb = j8 >> 3, ch = j8 & 7;
            *reinterpret_cast<uint4*>(Qs + kb * Cfg::Q_KB + (c >> 3) * 1024 + (c & 7) * 128 +
                                      ((ch ^ (c & 7)) << 4)) = v;
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    if (warp == Cfg::PRODUCER) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0)
            attn_produce<NST, DCH>(a, &kmap, &vmap, ring, full, empty, abort_flag, lb, kvh, t0, ntiles);
        __syncwarp();
    } else if (warp == Cfg::MMAW) {
        // ---------------------------------------------------------------- MMA issue
        constexpr uint32_t IDESC = umma_idesc_bf16(128, 128);
        const uint32_t sQ = smem_u32(Qs), sR = smem_u32(ring);
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        auto qk = [&](int j) {
            const int buf = j & 1;
            // the buffer's previous tile (j - 2): its P has been read by its P·V
            if (j >= 2 && !pwait_warp(&pv_done[buf], uint32_t((j - 2) >> 1) & 1u, abort_flag, a.status)) {
                ok = false;
                return;
            }
            tc_fence_after();
            for (int c = 0; c < DCH; ++c) {
                if (!pwait_warp(&full[stage], ph, abort_flag, a.status)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint64_t da = umma_desc_sw128(sQ + 2 * c * Cfg::Q_KB);
                const uint64_t db = umma_desc_sw128(sR + stage * Cfg::CHUNK);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16_warp(tbase + Cfg::TM_S + buf * 128,
                                       da + uint64_t((kb * Cfg::Q_KB + ks * 32) >> 4),
                                       db + uint64_t((kb * 16384 + ks * 32) >> 4), IDESC,
                                       (c | kb | ks) ? 1u : 0u);
                umma_commit_warp(&empty[stage]);
                if (++stage == NST) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            umma_commit_warp(&s_full[buf]);
        };
        auto pv = [&](int j) {
            const int buf = j & 1;
            if (!pwait_warp(&p_full[buf], uint32_t(j >> 1) & 1u, abort_flag, a.status)) {
                ok = false;
                return;
            }
            tc_fence_after();
            for (int c = 0; c < DCH; ++c) {
                if (!pwait_warp(&full[stage], ph, abort_flag, a.status)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint64_t db = umma_desc_sw128(sR + stage * Cfg::CHUNK);
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16_ts_warp(tbase + Cfg::TM_O + c * 128,
                                          tbase + Cfg::TM_S + buf * 128 + (kb * 4 + ks) * 8,
                                          db + uint64_t((kb * 16384 + ks * 32) >> 4), IDESC,
                                          (j > 0 || kb || ks) ? 1u : 0u);
                umma_commit_warp(&empty[stage]);
                if (++stage == NST) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            umma_commit_warp(&pv_done[buf]);
        };
        // the ring order: K(0), K(1), V(0), K(2), V(1), ...
        qk(0);
        if (ntiles > 1 && ok) qk(1);
        for (int j = 0; j < ntiles && ok; ++j) {
            pv(j);
            if (ok && j + 2 < ntiles) qk(j + 2);
        }
        umma_commit_warp(fin);          // arrives once every MMA issued above has completed
    } else {
        // ---------------------------------------------------------------- softmax warps
        // thread = (query row = TMEM lane, key half hf). Per tile: its 64 scores; the lazy maximum
        // (it moves only when the tile holds a score more than 8 above it: then the two threads
        // of the row exchange their tile maxima, take the same new maximum, and rescale O, each
        // half of its columns, and their partial sums); its weights rounded to bf16 over its half
        // of the packed P columns, and the sum of its rounded weights.
        const int q4 = warp & 3, hf = warp >> 2;
        const int row = q4 * 32 + lane;
        const uint32_t lane_off = uint32_t(q4 * 32) << 16;
        const int pbar = 1 + q4;                     // named barrier of the quarter's two warps
        const float sl2 = a.sl2;
        const int mylim = n0 + (row < a.nq ? row / G : T - 1);   // the last key the row may see
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int buf = j & 1;
            const int nvis = mylim - (t0 + j) * 128 - 64 * hf + 1;   // keys k < nvis of my half
            ok = pwait(&s_full[buf], uint32_t(j >> 1) & 1u, abort_flag, a.status) && ok;
            tc_fence_after();
            const uint32_t tS = tbase + lane_off + Cfg::TM_S + buf * 128;
            float s[64];
            {
                uint32_t r0[32], r1[32];
                tmem_ld32_nw(tS + 64 * hf, r0);
                tmem_ld32_nw(tS + 64 * hf + 32, r1);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    s[k] = __uint_as_float(r0[k]) * sl2;
                    s[32 + k] = __uint_as_float(r1[k]) * sl2;
                }
            }
            float mh[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < 64; ++k) mh[k & 3] = k < nvis ? fmaxf(mh[k & 3], s[k]) : mh[k & 3];
            const float mhalf = fmaxf(fmaxf(mh[0], mh[1]), fmaxf(mh[2], mh[3]));
            // both halves' S read (P may overwrite it); does any row of the quarter move?
            if (named_bar_or(pbar, 64, mhalf > m + 8.f)) {
                xch[hf * NQ + row] = mhalf;
                named_bar(pbar, 64);
                const float mt = fmaxf(xch[row], xch[NQ + row]);
                named_bar(pbar, 64);                 // both read before the next exchange
                const bool up = mt > m + 8.f;        // never for mt = -inf; the same in both
              if (__any_sync(0xffffffffu, up)) {
                const float al = up ? ((m == -INFINITY) ? 0.f : ex2(m - mt)) : 1.f;
                if (up) {
                    l *= al;
                    m = mt;
                }
                if (j > 0) {
                    // O holds P·V up to tile j-1: that product must be done first
                    ok = pwait(&pv_done[(j - 1) & 1], uint32_t((j - 1) >> 1) & 1u, abort_flag,
                               a.status) && ok;
                    tc_fence_after();
#pragma unroll 1
                    for (int c2 = 0; c2 < D / 64; ++c2) {
                        const uint32_t tO = tbase + lane_off + Cfg::TM_O + hf * (D / 2) + 32 * c2;
                        float o[32];
                        tmem_ld32(tO, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= al;
                        tmem_st32(tO, o);
                    }
                    tmem_wait_st();
                }
              }
            }
            float pk[32];
            float lp[2] = {0.f, 0.f};
#pragma unroll
            for (int k2 = 0; k2 < 32; ++k2) {
                const float e0 = 2 * k2 < nvis ? ex2(s[2 * k2] - m) : 0.f;
                const float e1 = 2 * k2 + 1 < nvis ? ex2(s[2 * k2 + 1] - m) : 0.f;
                const __nv_bfloat162 p2 = __floats2bfloat162_rn(e0, e1);     // e0 in the low half
                lp[k2 & 1] += __low2float(p2) + __high2float(p2);
                pk[k2] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&p2));
            }
            l += lp[0] + lp[1];
            tmem_st32(tS + 32 * hf, pk);                 // packed columns of keys 64 hf ..
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[buf]);
        }
        // ---------------------------------------------------------------- epilogue
        ok = pwait(&pv_done[(ntiles - 1) & 1], uint32_t((ntiles - 1) >> 1) & 1u, abort_flag,
                   a.status) && ok;
        tc_fence_after();
        named_bar(pbar, 64);                         // the last tile's maxima have been read
        xch[hf * NQ + row] = l;
        named_bar(pbar, 64);
        const float lrow = xch[row] + xch[NQ + row];
        if (!__any_sync(0xffffffffu, !ok)) {
            const bool mine = row < a.nq;
            const size_t ws_row = attn_ws_row(a, wk) + row;
            const int i = row / G, g = row - i * G;
            __nv_bfloat16* op = a.out + ((size_t(lb) * T + i) * a.Hq + kvh * G + g) * D + hf * (D / 2);
#pragma unroll 1
            for (int c2 = 0; c2 < D / 64; ++c2) {
                float o[32];
                tmem_ld32(tbase + lane_off + Cfg::TM_O + hf * (D / 2) + 32 * c2, o);
                if (!mine) continue;
                if (wk.whole) {
#pragma unroll
                    for (int k8 = 0; k8 < 4; ++k8) {
                        uint32_t w4[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[8 * k8 + 2 * h] / lrow,
                                                                            o[8 * k8 + 2 * h + 1] / lrow);
                            w4[h] = *reinterpret_cast<const uint32_t*>(&v2);
                        }
                        *reinterpret_cast<uint4*>(op + 32 * c2 + 8 * k8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else {
                    float* wo = a.ws_o + ws_row * D + hf * (D / 2) + 32 * c2;
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        *reinterpret_cast<float4*>(wo + 4 * k4) =
                            make_float4(o[4 * k4], o[4 * k4 + 1], o[4 * k4 + 2], o[4 * k4 + 3]);
                }
            }
            if (!wk.whole && mine && hf == 0) {
                float* ml = a.ws_ml + ws_row * 2;
                ml[0] = m;
                ml[1] = lrow;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == Cfg::MMAW) {
        tc_fence_after();
        if (!mbar_wait_bounded(fin, 0)) set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     ::"r"(tbase), "r"(uint32_t(Cfg::TM_COLS)));
    }
}

// ------------------------------------------------------------------ split merge
// block (tail unit, group of kCombRows query rows), thread = d; the partials of split s are at
// row (s · n_tail + tail) · nq. A split that saw no key has sum 0 and an unwritten O (read, never
// used).
constexpr int kCombRows = 8;
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
    const int tail = blockIdx.x, unit = a.n_full + tail, d = threadIdx.x;
    const int c0 = blockIdx.y * kCombRows;
    const size_t n_tail = size_t(a.units - a.n_full);
    const int kvh = unit % a.Hkv, lb = unit / a.Hkv, b = lb % a.B;
    const int n0 = __ldg(a.kv_len + b);
    if (n0 < 0 || n0 > a.ctx - a.T) return;
    const size_t sstride = n_tail * a.nq;                  // rows between splits
    const float2* mlp = reinterpret_cast<const float2*>(a.ws_ml);
    float mstar[kCombRows], num[kCombRows], den[kCombRows];
#pragma unroll
    for (int r = 0; r < kCombRows; ++r) { mstar[r] = -INFINITY; num[r] = 0.f; den[r] = 0.f; }
    const int nr = min(kCombRows, a.nq - c0);
    for (int s = 0; s < a.splits; ++s) {
        const size_t row0 = s * sstride + size_t(tail) * a.nq + c0;
#pragma unroll
        for (int r = 0; r < kCombRows; ++r) {
            if (r < nr) {
                const float2 ml = mlp[row0 + r];
                mstar[r] = ml.y > 0.f ? fmaxf(mstar[r], ml.x) : mstar[r];
            }
        }
    }
    for (int s = 0; s < a.splits; ++s) {
        const size_t row0 = s * sstride + size_t(tail) * a.nq + c0;
        float2 ml[kCombRows];
        float o[kCombRows];
#pragma unroll
        for (int r = 0; r < kCombRows; ++r) {
            ml[r] = r < nr ? mlp[row0 + r] : make_float2(0.f, 0.f);
            o[r] = r < nr ? a.ws_o[(row0 + r) * a.D + d] : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kCombRows; ++r) {
            if (ml[r].y > 0.f) {
                const float w = ex2(ml[r].x - mstar[r]);
                num[r] = fmaf(w, o[r], num[r]);
                den[r] = fmaf(w, ml[r].y, den[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kCombRows; ++r) {
        if (r < nr) {
            const int c = c0 + r, i = c / a.group, g = c - i * a.group;
            a.out[((size_t(lb) * a.T + i) * a.Hq + kvh * a.group + g) * a.D + d] =
                __float2bfloat16_rn(num[r] / den[r]);
        }
    }
}

// ------------------------------------------------------------------ truncation
__global__ void attn_truncate_kernel(int B, int T, const int32_t* n_acc, int32_t* kv_len,
                                     uint32_t* status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int n = n_acc[b];
    if (n < 0 || n > T) {
        set_status(status, GDN_STATUS_BAD_NACC);
        return;
    }
    kv_len[b] += n;
}

template <int D, int NQ>
static cudaError_t launch_attn_t(const AttnArgs& a, const CUtensorMap& kmap,
                                 const CUtensorMap& vmap, cudaStream_t s) {
    using Cfg = AttnCfg<D, NQ>;
    auto kern = attn_verify_kernel<D, NQ>;
    const cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), Cfg::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.n_full) + unsigned(a.units - a.n_full) * unsigned(a.splits), Cfg::NTHR,
           Cfg::SMEM, s>>>(a, kmap, vmap);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_attn_rows(const AttnArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, cudaStream_t s) {
    using Cfg = AttnRowsCfg<D>;
    auto kern = attn_rows_kernel<D>;
    const cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), Cfg::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<unsigned(a.n_full) + unsigned(a.units - a.n_full) * unsigned(a.splits), Cfg::NTHR,
           Cfg::SMEM, s>>>(a, kmap, vmap);
    return cudaGetLastError();
}

cudaError_t launch_attn_verify(const AttnArgs& a0, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t s) {
    AttnArgs a = a0;
    attn_append_kernel<<<dim3(a.B, a.L, a.Hkv), 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (a.nq > 64) {
        // 65-128 query rows per kv head: one CTA holds them all
        e = a.D == 128 ? launch_attn_rows<128>(a, kmap, vmap, s) : launch_attn_rows<256>(a, kmap, vmap, s);
        if (e != cudaSuccess || a.splits == 1 || a.units == a.n_full) return e;
        attn_combine_kernel<<<dim3(a.units - a.n_full, (a.nq + kCombRows - 1) / kCombRows), a.D, 0, s>>>(a);
        return cudaGetLastError();
    }
    const int nqp = a.nq <= 32 ? 32 : 64;
    if (a.D == 128)
        e = nqp == 32 ? launch_attn_t<128, 32>(a, kmap, vmap, s) : launch_attn_t<128, 64>(a, kmap, vmap, s);
    else
        e = nqp == 32 ? launch_attn_t<256, 32>(a, kmap, vmap, s) : launch_attn_t<256, 64>(a, kmap, vmap, s);
    if (e != cudaSuccess || a.splits == 1 || a.units == a.n_full) return e;
    attn_combine_kernel<<<dim3(a.units - a.n_full, (a.nq + kCombRows - 1) / kCombRows), a.D, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn_truncate(int B, int T, const int32_t* n_acc, int32_t* kv_len,
                                 uint32_t* status, cudaStream_t s) {
    attn_truncate_kernel<<<(B + 255) / 256, 256, 0, s>>>(B, T, n_acc, kv_len, status);
    return cudaGetLastError();
}

}  // namespace gdn
