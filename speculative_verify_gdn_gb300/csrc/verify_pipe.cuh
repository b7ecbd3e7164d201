// verify_pipe.cuh — persistent, warp-specialised gdn_verify for the Qwen3.6 head shape
// (Dk = Dv = 128, bf16 I/O, up to 2 value heads per key head; chains of T <= 16 positions, trees
// of T <= 32 nodes, and the fused rollback + verify for chains of T <= 8).
//
// Same computation as verify_impl.cuh (see its header for the method and the sources): per value
// head, P = S_0·[K|Q] in three TF32 products on tcgen05, the Gram block, and the per-row
// recurrence for δ and o. What changes is the schedule. One CTA per SM walks a sequence of key
// heads ("units": (layer, sequence, key head), each with its value heads) through warp roles that
// hand work to each other through mbarriers:
//
//   warp 0       state loader  2-D TMA of each state K-block (128 rows x 32 fp32 = 16 KiB) into a
//                              ring of shared-memory slots
//   warp 14      input loader  per part (q, k, each v): one 2-D TMA box of the conv-state rows, one
//                              of the unit's T qkv rows and one bulk copy of the conv taps (staging
//                              ring, 2 slots)
//   warps 6-9    convert       per K-block: S_hi = trunc_tf32(S) and S_lo = S − S_hi from the slot
//                              into a ring of TMEM slots (32 + 32 columns); the shared-memory slot is
//                              free as soon as it has been read
//   warp 1       mma           per K-block: S_hi·[X_hi ; X_lo] and S_lo·X_hi, both with A from TMEM,
//                              into separate accumulators; the unit's value heads (or, with one
//                              value head, even and odd K-steps) in turn, so that consecutive MMAs
//                              never update the same accumulator (2 unit slots of P in TMEM)
//   warps 2-5    prep          per unit: conv + SiLU, norms, the [X_hi ; X_lo] tile, the Gram block
//                              (mma.sync, 3xTF32) and each value head's coefficient records (for
//                              16-position chains the Gram block and records are the epilogue
//                              warps' first task, while the unit's products run)
//   warps 10-13  epilogue      per head: P rows from TMEM (sum of its partial accumulators),
//                              recurrence, o and δ stores
//
// The state stream is read from shared memory exactly once (by the convert warps: the tensor core
// takes both operand halves from TMEM), and a shared-memory slot is held only from its TMA until
// its K-block has been split, so the loader runs ahead of the unit prologue by the whole ring.
// Every wait is bounded: on a timeout the CTA records WAIT_TIMEOUT, the producers stop issuing, and
// the other roles run on without waiting (results are then garbage, never a hang). The pipeline
// waits give up after VerifyArgs::wait_ns (default one second; gdn_set_wait_limit_ns); the drains
// before the CTA exits (copies in flight, MMAs before TMEM is released) keep the full second.
//
// COMMIT (gdn_rollback_verify): the same pass first commits the previous round's accepted steps,
// as gdn_rollback does ("GDN investigation" §4, tape replay), then verifies the new round from the
// committed state. With n = n_acc_prev[b], c_s = Γ(s+1 .. n-1), Γ = Γ(0 .. n-1) and the rank-n
// term A Kᵀ (A[i][s] = c_s δ_s[i], K[j][s] = k_s[j] of the previous round):
//     S_n = Γ · S_0 + A Kᵀ,        S_n · X = Γ · (S_0 · X) + A · (Kᵀ X).
// So the tensor-core products still run on the loaded S_0; the epilogue forms Kᵀ X (n x 2T,
// mma.sync) and applies Γ and A · (Kᵀ X) to each P row. For the write-back the convert warps form
// S_n = Γ S_0 + A Kᵀ of each K-block in shared memory with warp-level mma.sync (3xTF32, K = 8) and
// a store warp (warp 15) writes it back by TMA store. The conv window is the last W-1 rows of (old
// conv state ++ the previous round's accepted raw rows), staged from both buffers; the prep warps
// stash those rows and the epilogue writes them out as the new conv state. So each state tile is
// read once and written once per round, instead of read by verify, read and written by rollback.
//
// GDK (one decay per key channel, g [L][B][T][Hv][Dk]; chains of T <= 8): the decay of S_0 up to
// step t is a per-column factor, so each value head has its own B tile [A_t ⊙ k_t ; A_t ⊙ q_t]
// (A_t[c] = Π_{r≤t} a_r[c]) and the MMAs of head j read tile j; the Gram entries carry the decay
// of each column between write s and read t, CK[t][s] = Σ_c k_s[c] k_t[c] Π_{s<r≤t} a_r[c] (CQ
// with q_t), built by the epilogue warps as running products (never a ratio of cumulative
// products, so a zero gate stays exact); the recurrence then runs with γ = c0 = 1.
//
// TREE: node v's products come from the same S_0 · [K|Q] through the ancestor-sum identity
// (S_p k_v = Γ(root→p) S_0 k_v + Σ_{a ancestor of v} Γ(a→p) δ_a (k_a·k_v), the same with q_v): the
// coefficient records hold Γ(a→p) times the Gram entry for ancestors and zero elsewhere, and each
// node's conv window is itself, its nearest ancestors, then the conv state's rows. The B tile keeps
// raw q, k; the inverse norms go into the coefficients. T = 32 (BIG) keeps one B-tile / meta slot:
// the next unit's prep starts once this unit's products are done and waits for this unit's
// epilogue only before writing its records; the epilogue warps compute v into TMEM themselves and
// solve each value head's recurrence as one triangular system on the tensor core (the rows of
// (I + diag(βγ) CK)⁻¹ by back-substitution along each node's root path, then one product for all
// 128 value rows).
#pragma once

#include "verify_impl.cuh"

namespace gdn {

template <typename IO, int TMAX, int G, bool COMMIT, bool TREE, bool GDK = false>
struct PipeCfg {
    static constexpr int D = 128, KB = 4, ES = int(sizeof(IO)), TMAX_ = TMAX;
    // B tiles per unit slot: one per value head with per-key-channel gates, else one shared
    static constexpr int NXT = GDK ? G : 1;
    // T up to 32 (trees): one slot each for the B tile, the records and the staging (the next
    // unit's prep overlaps this unit's epilogue; see the kernel), one accumulator per chain
    static constexpr bool BIG = TMAX >= 32;
    static constexpr int NXS = BIG ? 1 : 2;                  // B-tile / meta slots
    static constexpr int NSS = BIG ? 1 : 2;                  // staging slots
    static constexpr int NWARP = COMMIT ? 16 : 15, NTHR = 32 * NWARP;
    static constexpr int NP = 2 * TMAX < 16 ? 16 : 2 * TMAX;
    static constexpr int XROWS = 2 * NP, XKB = XROWS * 128, X_BYTES = KB * XKB;
    static constexpr int KSLOT = 128 * 128;                 // one state K-block: 128 rows x 128 B
    // accumulator chains per value head: with one value head per unit, even and odd K-steps go to
    // separate accumulators, so every unit has two chains to alternate with
    static constexpr int S = G == 1 ? 2 : 1;
    // TMEM: NUS unit slots of 2 chains x (hi pass: 2NP columns at +0, lo pass: NP columns at
    // +2NP; 32-aligned — or, BIG, one NP-column accumulator that all three products add into),
    // then a ring of NTS K-block slots (hi 32 + lo 32 columns); BIG: then the conv outputs v of
    // the unit's value heads, column j TMAX + t, lane = value row (written by the epilogue warps)
    static constexpr int TMEM_COLS = 512;
    static constexpr int CH_COLS = BIG ? NP : (3 * NP + 31) / 32 * 32, P_COLS = 2 * CH_COLS;
    static constexpr int NUS = TMAX <= 8 ? 2 : 1;
    static constexpr int T_RING = NUS * P_COLS;
    static constexpr int V_COLS = BIG ? G * TMAX : 0;
    // BIG: the epilogue's triangular solve on the tensor core: its A operand r (hi 32 + lo 32
    // columns) at T_R, its accumulator [δ | o] (64 columns) at T_D, both 64-column aligned ahead of v
    static constexpr int UT_COLS = BIG ? 128 : 0;
    static constexpr int NTS_FIT = (TMEM_COLS - T_RING - V_COLS - UT_COLS) / 64;
    static constexpr int NTS = NTS_FIT < 4 ? NTS_FIT : 4;
    static constexpr int T_R = T_RING + NTS * 64, T_D = T_R + 64, T_V = T_R + UT_COLS;
    static constexpr int NPARTS = 2 + G;                     // q, k, v of each value head
    // staged rows per part (W <= 4): W-1 old conv-state rows, the T qkv rows and, when committing,
    // W-1 rows of the previous round's qkv ending at its accepted count
    static constexpr int NRMAX = 3 + TMAX + (COMMIT ? 3 : 0);
    static constexpr int RAW_BYTES = NPARTS * NRMAX * D * ES + NPARTS * D * 4 * ES;
    // (BIG: a 1024-byte multiple, so the meta slot after it starts on a swizzle-atom boundary)
    static constexpr int STAGE_BYTES = BIG ? (RAW_BYTES + 1023) / 1024 * 1024 : (RAW_BYTES + 127) / 128 * 128;
    // meta slot (floats): per value head j and position t a record {c0, γ, β, k_t·q_t, (TREE)
    // c0q, group mask, 0, 0, CK[TMAX], CQ[TMAX]} (16-byte aligned), the conv outputs V[G][TMAX][D]
    // and, COMMIT, GP[s][c] = k'_s·X_c of the previous round's k'_s and the new conv-state rows
    // CW[NPARTS][3][D] (io type). Trees keep raw (unnormalised) q, k in the B tile: c0 and c0q
    // carry 1/|k_t| and 1/|q_t|, and bit g of the mask is set when CK / CQ entries 4g .. 4g+3 can
    // be nonzero (ancestors only).
    // BIG (T = 32 trees) uses per-head blocks instead: CK and CQ transposed ([x][t], zero for
    // non-ancestors) of each head (M_REC, RJ apart), a 16 KiB operand tile (M_UT), then the fields
    // c0k, c0q, γ, β, k·q [5][TMAX] of each head (M_FLD, FJ apart), the unit's parents [TMAX] (ints,
    // M_PAR; -1 past T). The epilogue turns CK, CQ into
    // the solve's B operand [M | N] (64 rows x 32 fp32, hi rows then lo rows, 128-byte swizzle):
    // head 0's into M_UT, head 1's over the CK / CQ blocks once every thread has read them.
    static constexpr int HDR = TREE ? 8 : 4;
    static constexpr int RS = HDR + 2 * TMAX;
    static constexpr int RJ = BIG ? 2 * TMAX * TMAX : TMAX * RS;
    static constexpr int F_CKT = 0, F_CQT = TMAX * TMAX;
    static constexpr int F_C0K = 0, F_C0Q = TMAX, F_GAM = 2 * TMAX, F_BET = 3 * TMAX, F_KQ = 4 * TMAX,
                         FJ = 5 * TMAX;
    static constexpr int UT_FLOATS = BIG ? 2 * 64 * 32 : 0;
    // BIG keeps v in TMEM; its meta slot holds the Gram block [TMAX][2 TMAX] instead (M_V)
    // GDK: then the plain normalised rows k_t, q_t [2 TMAX][D] for the epilogue's Gram (M_XP)
    static constexpr int M_REC = 0, M_UT = G * RJ, M_FLD = M_UT + UT_FLOATS, M_PAR = M_FLD + (BIG ? G * FJ : 0),
                         M_V = M_PAR + (BIG ? TMAX : 0),
                         M_GP = M_V + (BIG ? 2 * TMAX * TMAX : G * TMAX * D),
                         M_CW = M_GP + (COMMIT ? 2 * TMAX * TMAX : 0),
                         M_XP = M_CW + (COMMIT ? (NPARTS * 3 * D * ES + 3) / 4 : 0),
                         M_FLOATS = M_XP + (GDK ? 2 * TMAX * D : 0);
    static constexpr int META_BYTES = (M_FLOATS * 4 + 127) / 128 * 128;
    // commit slot (floats): previous round's k_s rows [TMAX][D], δ_s rows [G][TMAX][D],
    // c_s = Γ(s+1 .. n-1) [G][TMAX], Γ(0 .. n-1) [G]
    // k and δ rows padded to 136 floats: the convert warps' fragment loads (row = lane & 3 or
    // its +4, column / state row ~ lane >> 2) fall in distinct banks
    static constexpr int KP_KS = D + 8;
    static constexpr int KP_K = 0, KP_DL = TMAX * KP_KS, KP_C = KP_DL + G * TMAX * KP_KS,
                         KP_GAM = KP_C + G * TMAX, KP_FLOATS = KP_GAM + 4;
    static constexpr int KP_BYTES = COMMIT ? (KP_FLOATS * 4 + 127) / 128 * 128 : 0;
    // Gram block X_m · k_n (m < 2 TMAX, n < TMAX) in 16 x 8 mma.sync tiles: one tile (TMAX <= 8)
    // split over the 4 prep warps by channels, or 4 / 16 tiles (TMAX = 16 / 32), a quarter per warp
    static constexpr int GRAM_TILES = ((2 * TMAX + 15) / 16) * ((TMAX + 7) / 8);
    // prep scratch (floats): norm partials [4][2TMAX] (chains), inverse norms [2TMAX], Gram partials
    // [4 warps][16][8] (one-tile case), Gram [TMAX][2TMAX] (BIG: in the meta slot instead),
    // tree parents [TMAX] and conv-window offsets [TMAX][4] (ints)
    // (COMMIT) epilogue: partials of k'_s · X_c [4 warps][16][8]
    static constexpr int S_NRM = 0, S_INV = S_NRM + (TREE ? 0 : 8 * TMAX), S_GP = S_INV + 2 * TMAX,
                         S_GRAM = S_GP + (GRAM_TILES == 1 ? 4 * 128 : 0),
                         S_PAR = S_GRAM + (BIG ? 0 : 2 * TMAX * TMAX), S_WIN = S_PAR + (TREE ? TMAX : 0),
                         S_EGP = S_WIN + (TREE ? 4 * TMAX + 4 : 0),
                         S_FLOATS = S_EGP + (COMMIT ? 4 * 128 : 0);
    // shared-memory K-block ring: as many 16 KiB slots as the rest leaves room for (at most 8)
    static constexpr size_t REST = NXS * NXT * size_t(X_BYTES) + NSS * size_t(STAGE_BYTES) + NXS * size_t(META_BYTES) +
                                   2 * size_t(KP_BYTES) + size_t(S_FLOATS) * 4 + 64 * 8 + 16 + 16 + 1024;
    static constexpr int NKS_FIT = int((227 * 1024 - REST) / KSLOT);
    static constexpr int NKS = NKS_FIT > 8 ? 8 : NKS_FIT;

    static constexpr size_t OFF_RING = 0;
    static constexpr size_t OFF_X = OFF_RING + size_t(NKS) * KSLOT;
    static constexpr size_t OFF_STAGE = OFF_X + NXS * NXT * size_t(X_BYTES);
    static constexpr size_t OFF_META = OFF_STAGE + NSS * size_t(STAGE_BYTES);
    static constexpr size_t OFF_KP = OFF_META + NXS * size_t(META_BYTES);
    static constexpr size_t OFF_SCR = OFF_KP + 2 * size_t(KP_BYTES);
    static constexpr size_t OFF_BAR = (OFF_SCR + size_t(S_FLOATS) * 4 + 15) / 16 * 16;
    static constexpr int NBAR = 3 * NKS + 2 * NTS + 8 * 2 + 3 + 2 + 2;
    static constexpr size_t OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM base, abort flag
    static constexpr size_t SMEM = OFF_MISC + 16 + 1024;

    static_assert(T_V + V_COLS <= TMEM_COLS && NTS >= G, "TMEM budget");
    static_assert(!BIG || (OFF_META % 1024 == 0 && (M_UT * 4) % 1024 == 0 && (M_FLD * 4) % 16 == 0),
                  "the solve's B tiles need 1024-byte bases");
    static_assert(NKS >= 2 * G, "shared-memory ring");
    static_assert(G * S == 2, "two accumulator chains per unit");
    static_assert(!COMMIT || TMAX <= 8, "the fused rollback serves T <= 8");
    static_assert(!(COMMIT && TREE), "the fused rollback serves chains");
    static_assert(!BIG || TREE, "T = 32 is the tree workload's size");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(OFF_X % 1024 == 0 && X_BYTES % 1024 == 0, "swizzle atoms need 1024-byte bases");
    static_assert((RS * 4) % 16 == 0 && (RJ * 4) % 16 == 0 && (M_V * 4) % 16 == 0 && (M_GP * 4) % 16 == 0 &&
                  (M_CW * 4) % 16 == 0, "records are read as float4, CW rows as 16-byte vectors");
    static_assert((KP_DL * 4) % 16 == 0 && (KP_KS * 4) % 16 == 0, "bulk-copy destinations");
    static_assert(GRAM_TILES == 1 || GRAM_TILES % 4 == 0, "Gram block: one tile, or a quarter per prep warp");
    static_assert(!GDK || (!TREE && !COMMIT && TMAX <= 8), "per-key-channel gates: chains of T <= 8");
};

// D[tmem] (+)= A[tmem] · B[smem descriptor]ᵀ, kind::tf32. Called by a whole converged warp with
// warp-uniform operands; one elected lane issues. (Issue from a lone diverged lane costs about three
// times as many cycles per MMA as the tensor core needs for these small shapes.)
__device__ __forceinline__ void umma_tf32_ts_warp(uint32_t dtmem, uint32_t atmem, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(dtmem), "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ldmatrix with 16-bit 8 x 8 matrices on fp32 data: each lane receives the 32-bit word (row
// lane / 4, word lane % 4) of each matrix, which are the m16n8k8 tf32 fragment positions. Lanes
// 8j .. 8j+7 give the 16-byte row addresses of matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// shared -> global copies of the async proxy, tracked in the issuing thread's bulk groups
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(src))
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
          "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
          "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// warp-level D(16x8) += A(16x8) · B(8x8), TF32 operands (already truncated), fp32 accumulate
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&av)[4], uint32_t b0,
                                                uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(av[0]), "r"(av[1]), "r"(av[2]), "r"(av[3]), "r"(b0), "r"(b1));
}

// 1/sqrt(s) for s > 0: the hardware approximation refined by one Newton-Raphson step
// (y <- y (3 - s y^2) / 2), a few ulp from the correctly rounded value
__device__ __forceinline__ float inv_sqrt_nr(float s) {
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(s));
    return y * fmaf(-0.5f * s * y, y, 1.5f);
}

// p + n, hidden from the compiler's address arithmetic: a fully unrolled loop of stores then
// advances one pointer instead of holding every iteration's 64-bit address in registers
template <typename P>
__device__ __forceinline__ P* opaque_advance(P* p, size_t n) {
    P* q = p + n;
    asm volatile("" : "+l"(q));
    return q;
}

// global stores under a predicate, without a branch (unrolled loops stay one basic block)
__device__ __forceinline__ void st_global_if(float* p, float v, bool c) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.f32 [%0], %1;\n\t}"
                 ::"l"(__cvta_generic_to_global(p)), "f"(v), "r"(int(c)));
}
__device__ __forceinline__ void st_global_if(__nv_bfloat16* p, float v, bool c) {
    const unsigned short h = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.b16 [%0], %1;\n\t}"
                 ::"l"(__cvta_generic_to_global(p)), "h"(h), "r"(int(c)));
}
__device__ __forceinline__ void st_global_if(float* p, float4 v, bool c) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t@q st.global.v4.f32 [%0], {%1, %2, %3, %4};\n\t}"
                 ::"l"(__cvta_generic_to_global(p)), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(int(c)));
}

// two bf16 values packed in a 32-bit word (element 0 in the low half) to floats (exact)
__device__ __forceinline__ float bf2_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf2_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Tree conv + SiLU of NPH consecutive parts (from part0, all of them q / k when TO_X, all v
// heads otherwise) over channels c2, c2 + 1 for every node: node t's window is the staged rows at
// element offsets win[4 t + d] (tap d = distance d). Nodes go in groups: every load of a group is
// issued before any store, so the loads overlap instead of queueing behind the previous node's
// stores; the loop body has no branch. q (part 0) and k (part 1) go to B-tile rows TMAX + t and
// t with their tf32 remainders at NP + row; v heads to the meta slot.
template <typename Cfg, int NPH, bool TO_X, typename IO>
__device__ __forceinline__ void tree_conv_parts(int part0, int c2, const IO* qs, const IO* cws, int NR,
                                                int W, int T, const int* win, unsigned char* Xb,
                                                float* meta) {
    constexpr int TMAX = Cfg::TMAX_, D = Cfg::D, NP = Cfg::NP, XKB = Cfg::XKB;
    constexpr int NB = NPH == 1 ? 8 : 4;                 // nodes per group
    static_assert(sizeof(IO) == 2, "the tree conv reads bf16 pairs");
    float wr[NPH][4][2];
    const IO* col[NPH];
    int rbase[NPH];
#pragma unroll
    for (int k = 0; k < NPH; ++k) {
        const int part = part0 + k;
        const IO* wp = cws + (size_t(part) * D + c2) * W;
#pragma unroll
        for (int d = 0; d < 4; ++d)
#pragma unroll
            for (int c = 0; c < 2; ++c) wr[k][d][c] = d < W ? io_to_f(wp[c * W + W - 1 - d]) : 0.f;
        col[k] = qs + size_t(part) * NR * D + c2;
        rbase[k] = TO_X ? (part == 0 ? TMAX : 0) : (part - 2) * TMAX;
    }
    const int4* win4 = reinterpret_cast<const int4*>(win);
#pragma unroll 1
    for (int t0 = 0; t0 < TMAX; t0 += NB) {
        uint32_t u[NB][NPH][4];
#pragma unroll
        for (int tb = 0; tb < NB; ++tb) {
            const int4 w4 = win4[t0 + tb];
            const int src[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < NPH; ++k)
#pragma unroll
                for (int d = 0; d < 4; ++d) u[tb][k][d] = *reinterpret_cast<const uint32_t*>(col[k] + src[d]);
        }
#pragma unroll
        for (int tb = 0; tb < NB; ++tb) {
            const int t = t0 + tb;
#pragma unroll
            for (int k = 0; k < NPH; ++k) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int d = 3; d >= 0; --d) {
                    a0 = fmaf(wr[k][d][0], bf2_lo(u[tb][k][d]), a0);
                    a1 = fmaf(wr[k][d][1], bf2_hi(u[tb][k][d]), a1);
                }
                const float y0 = t < T ? silu_fast(a0) : 0.f, y1 = t < T ? silu_fast(a1) : 0.f;
                const int r = rbase[k] + t;
                if constexpr (TO_X) {
                    *reinterpret_cast<float2*>(Xb + sw128_off(r, c2, XKB)) = make_float2(y0, y1);
                    *reinterpret_cast<float2*>(Xb + sw128_off(NP + r, c2, XKB)) =
                        make_float2(y0 - tf32_trunc(y0), y1 - tf32_trunc(y1));
                } else {
                    *reinterpret_cast<float2*>(meta + Cfg::M_V + r * D + c2) = make_float2(y0, y1);
                }
            }
        }
    }
}

// Tree conv + SiLU of the v heads for value row i (the calling thread's TMEM lane): head j, node
// t goes to TMEM column tv + j TMAX + t. Groups of 16 nodes: loads first, then math, then one
// 16-column store.
template <typename Cfg, typename IO>
__device__ __forceinline__ void tree_vconv_tmem(int i, const IO* qs, const IO* cws, int NR, int W, int T,
                                                const int* win, uint32_t tv) {
    constexpr int TMAX = Cfg::TMAX_, D = Cfg::D, G = Cfg::NPARTS - 2;
    const int4* win4 = reinterpret_cast<const int4*>(win);
#pragma unroll 1
    for (int j = 0; j < G; ++j) {
        const IO* wp = cws + (size_t(2 + j) * D + i) * W;
        float wr[4];
#pragma unroll
        for (int d = 0; d < 4; ++d) wr[d] = d < W ? io_to_f(wp[W - 1 - d]) : 0.f;
        const IO* col = qs + size_t(2 + j) * NR * D + i;
#pragma unroll 1
        for (int t0 = 0; t0 < TMAX; t0 += 16) {
            float x[16][4];
#pragma unroll
            for (int tb = 0; tb < 16; ++tb) {
                const int4 w4 = win4[t0 + tb];
                x[tb][0] = io_to_f(col[w4.x]);
                x[tb][1] = io_to_f(col[w4.y]);
                x[tb][2] = io_to_f(col[w4.z]);
                x[tb][3] = io_to_f(col[w4.w]);
            }
            uint32_t y[16];
#pragma unroll
            for (int tb = 0; tb < 16; ++tb) {
                float acc = 0.f;
#pragma unroll
                for (int d = 3; d >= 0; --d) acc = fmaf(wr[d], x[tb][d], acc);
                y[tb] = __float_as_uint(t0 + tb < T ? silu_fast(acc) : 0.f);
            }
            tmem_st16(tv + j * TMAX + t0, y);
        }
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Gram block and coefficient records of a chain unit (the epilogue warps run this for chains of
// 16 positions, where the prep warps are the busiest role; the prep warps run the same code for
// the other shapes): 128 threads, w4 = warp in the group, t128 = thread in the group, named
// barrier `bar` among them.
template <typename Cfg>
__device__ __forceinline__ void chain_gram_fold(int w4, int lane, int t128, int bar, int T,
                                                const unsigned char* Xb, float* meta, float* gram,
                                                float* gp) {
    constexpr int TMAX = Cfg::TMAX_, G = Cfg::NPARTS - 2, RS = Cfg::RS, XKB = Cfg::XKB;
    const int gq = lane >> 2, gt4 = lane & 3;
    // Gram block on the warp tensor path: D[m][n] = X_m · k_n, 3xTF32 (hi·hi + hi·lo + lo·hi);
    // rows m: k_0.., q_0.. (zero beyond 2 TMAX). One 16 x 8 tile: each warp takes 32 channels
    // and the partials are summed; four tiles (TMAX = 16): warp w4 takes tile w4, all channels.
    if constexpr (Cfg::GRAM_TILES >= 4) {
      // a warp's tiles (one, or four sharing the column block k_{8 w4 ..}) in one pass over
      // the channels, hi·hi + lo·hi and hi·lo in separate accumulators: 2 TPW independent
      // chains
      constexpr int NTN = (TMAX + 7) / 8, TPW = Cfg::GRAM_TILES / 4;
      static_assert(TPW == 1 || NTN == 4, "a warp's tiles share their column block");
      const int nt = w4 % NTN;
      // one tile per warp: four accumulator sets, rotated over the K-steps
      constexpr int NACC = TPW == 1 ? 4 : 1, KUNROLL = TPW == 1 ? 4 : 2;
      float acc[TPW * NACC][4], acl[TPW * NACC][4];
#pragma unroll
      for (int m = 0; m < TPW * NACC; ++m)
#pragma unroll
          for (int e = 0; e < 4; ++e) { acc[m][e] = 0.f; acl[m][e] = 0.f; }
#pragma unroll (KUNROLL)
      for (int ks = 0; ks < 16; ++ks) {
        const int ka = NACC == 1 ? 0 : (ks & 3);
        // B: rows 8 nt .., channels 8 ks + 0..3 and + 4..7 (ldmatrix, lanes 0..15)
        uint32_t rb[2];
        ldsm_x2(smem_u32(Xb + sw128_off(8 * nt + (lane & 7), 8 * ks + ((lane >> 3) & 1) * 4, XKB)), rb);
        const float bv0 = __uint_as_float(rb[0]), bv1 = __uint_as_float(rb[1]);
        const float bh0 = tf32_trunc(bv0), bh1 = tf32_trunc(bv1);
        const uint32_t bl0 = __float_as_uint(tf32_trunc(bv0 - bh0));
        const uint32_t bl1 = __float_as_uint(tf32_trunc(bv1 - bh1));
        uint32_t ahi[TPW][4], alo[TPW][4];
#pragma unroll
        for (int m = 0; m < TPW; ++m) {
            const int mt = TPW == 1 ? w4 / NTN : m;
            // A: rows 16 mt + 0..7 / 8..15, channels 8 ks + 0..3 / 4..7 (ldmatrix)
            uint32_t ra[4];
            ldsm_x4(smem_u32(Xb + sw128_off(16 * mt + ((lane >> 3) & 1) * 8 + (lane & 7),
                                            8 * ks + (lane >> 4) * 4, XKB)), ra);
            const float av[4] = {__uint_as_float(ra[0]), __uint_as_float(ra[1]), __uint_as_float(ra[2]),
                                 __uint_as_float(ra[3])};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float h = tf32_trunc(av[e]);
                ahi[m][e] = __float_as_uint(h);
                alo[m][e] = __float_as_uint(tf32_trunc(av[e] - h));
            }
        }
#pragma unroll
        for (int m = 0; m < TPW; ++m) {
            mma_tf32_16x8x8(acc[m + ka], ahi[m], __float_as_uint(bh0), __float_as_uint(bh1));
            mma_tf32_16x8x8(acl[m + ka], ahi[m], bl0, bl1);
        }
#pragma unroll
        for (int m = 0; m < TPW; ++m)
            mma_tf32_16x8x8(acc[m + ka], alo[m], __float_as_uint(bh0), __float_as_uint(bh1));
      }
#pragma unroll
      for (int q2 = 1; q2 < NACC; ++q2)
#pragma unroll
          for (int e = 0; e < 4; ++e) { acc[0][e] += acc[q2][e]; acl[0][e] += acl[q2][e]; }
      // Gr[a][c] = k_a · X_c = D[c][a]
#pragma unroll
      for (int m = 0; m < TPW; ++m) {
        const int mt = TPW == 1 ? w4 / NTN : m;
        const int c0 = 16 * mt + gq, a0 = 8 * nt + 2 * gt4;
        gram[a0 * 2 * TMAX + c0] = acc[m][0] + acl[m][0];
        gram[(a0 + 1) * 2 * TMAX + c0] = acc[m][1] + acl[m][1];
        gram[a0 * 2 * TMAX + c0 + 8] = acc[m][2] + acl[m][2];
        gram[(a0 + 1) * 2 * TMAX + c0 + 8] = acc[m][3] + acl[m][3];
      }
    } else {
      {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const int ch = 32 * w4 + 8 * ks + gt4;
            float av[4];
            av[0] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch, XKB));
            av[2] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch + 4, XKB));
            av[1] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch, XKB)) : 0.f;
            av[3] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch + 4, XKB)) : 0.f;
            const float bv0 = gq < TMAX ? av[0] : 0.f, bv1 = gq < TMAX ? av[2] : 0.f;
            uint32_t ahi[4], alo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float h = tf32_trunc(av[e]);
                ahi[e] = __float_as_uint(h);
                alo[e] = __float_as_uint(tf32_trunc(av[e] - h));
            }
            const float bh0 = tf32_trunc(bv0), bh1 = tf32_trunc(bv1);
            const uint32_t bl0 = __float_as_uint(tf32_trunc(bv0 - bh0));
            const uint32_t bl1 = __float_as_uint(tf32_trunc(bv1 - bh1));
            mma_tf32_16x8x8(acc, ahi, __float_as_uint(bh0), __float_as_uint(bh1));
            mma_tf32_16x8x8(acc, ahi, bl0, bl1);
            mma_tf32_16x8x8(acc, alo, __float_as_uint(bh0), __float_as_uint(bh1));
        }
        float* g4 = gp + w4 * 128;
        g4[gq * 8 + 2 * gt4] = acc[0];
        g4[gq * 8 + 2 * gt4 + 1] = acc[1];
        g4[(gq + 8) * 8 + 2 * gt4] = acc[2];
        g4[(gq + 8) * 8 + 2 * gt4 + 1] = acc[3];
      }
      named_bar(bar, 128);
      {
        const int m = t128 >> 3, nn = t128 & 7;
        if (m < 2 * TMAX && nn < TMAX)
            gram[nn * 2 * TMAX + m] = gp[t128] + gp[128 + t128] + gp[256 + t128] + gp[384 + t128];
      }
    }
    named_bar(bar, 128);
    if constexpr (TMAX >= 16) {
    // per (value head, position v), walking back over x = v-1 .. 0: CK[v][x] =
    // Γ(x+1..v-1) k_x·k_v and CQ[v][x] = Γ(x+1..v-1) k_x·q_v; c0[v] = Γ(0..v-1), k_v·q_v
    for (int idx = t128; idx < G * TMAX; idx += 128) {
        const int fj = idx / TMAX, fv = idx - fj * TMAX;
        if (fv < T) {
            const float* hrec = meta + Cfg::M_REC + fj * TMAX * RS;     // γ at [y * RS + 1]
            float* rec = meta + Cfg::M_REC + idx * RS;
            float coef = 1.f;
            for (int fx = fv - 1; fx >= 0; --fx) {
                rec[4 + fx] = coef * gram[fx * 2 * TMAX + fv];
                rec[4 + TMAX + fx] = coef * gram[fx * 2 * TMAX + TMAX + fv];
                coef *= hrec[fx * RS + 1];
            }
            rec[0] = coef;
            rec[3] = gram[fv * 2 * TMAX + TMAX + fv];
        }
    }
    } else {
    // per value head, one thread per (v, x ≤ v): CK[v][x] = Γ(x→v-1) k_x·k_v and
    // CQ[v][x] = Γ(x→v-1) k_x·q_v for x < v; c0[v] = Γ(root→v-1) and k_v·q_v for x = v
    for (int idx = t128; idx < G * TMAX * TMAX; idx += 128) {
        const int fj = idx / (TMAX * TMAX), fv = (idx / TMAX) % TMAX, fx = idx % TMAX;
        if (fv < T && fx <= fv) {
            const float* hrec = meta + Cfg::M_REC + fj * TMAX * RS;     // γ at [y * RS + 1]
            float* rec = meta + Cfg::M_REC + (fj * TMAX + fv) * RS;
            const int y0 = fx < fv ? fx + 1 : 0;
            float coef = 1.f;
#pragma unroll
            for (int yy = 0; yy < TMAX - 1; ++yy)
                if (yy >= y0 && yy < fv) coef *= hrec[yy * RS + 1];
            if (fx < fv) {
                rec[4 + fx] = coef * gram[fx * 2 * TMAX + fv];
                rec[4 + TMAX + fx] = coef * gram[fx * 2 * TMAX + TMAX + fv];
            } else {
                rec[0] = coef;
                rec[3] = gram[fv * 2 * TMAX + TMAX + fv];
            }
        }
    }
    }
    named_bar(bar, 128);
}

// Gram block and coefficient records of a chain unit with one decay per key channel (the epilogue
// warps run it; 128 threads, t128 = thread in the group, named barrier `bar` among them). Thread
// (head j, write s, channel group c8) keeps w[m] = Π_{s<r≤t} a_r[c] for its channels c = c8 + 8m
// and walks t upward: CK[t][s] = Σ_c k_s[c] w[c] k_t[c], CQ[t][s] with q_t, summed over the 8
// lanes of the group. Also c0 = 1 (the decays of S_0 are in the B tiles) and k_s·q_s. `g_lb` is
// the unit's gates, g + (l B + b) T Hv D.
template <typename Cfg>
__device__ __forceinline__ void gdk_gram_records(int t128, int kh, int Hv, int T, int bar,
                                                 const float* g_lb, float* meta) {
    constexpr int TMAX = Cfg::TMAX_, G = Cfg::NPARTS - 2, RS = Cfg::RS, D = Cfg::D, NJ = D / 8;
    static_assert(TMAX <= 8 && G * TMAX * 8 <= 128, "one thread per (head, write, channel group)");
    const int j = t128 >> 6, s = (t128 >> 3) & 7, c8 = t128 & 7;
    const bool act = j < G && s < T;
    const int h = kh * G + (j < G ? j : 0);
    const float* XP = meta + Cfg::M_XP;
    float* recj = meta + Cfg::M_REC + (j < G ? j : 0) * TMAX * RS;
    float ks[NJ], w[NJ];
    float kq = 0.f;
#pragma unroll
    for (int m = 0; m < NJ; ++m) {
        const int c = c8 + 8 * m;
        w[m] = 1.f;
        ks[m] = act ? XP[s * D + c] : 0.f;
        kq = fmaf(ks[m], act ? XP[(TMAX + s) * D + c] : 0.f, kq);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
    if (c8 == 0 && act) {
        recj[s * RS + 0] = 1.f;
        recj[s * RS + 3] = kq;
    }
#pragma unroll 1
    for (int t = 1; t < TMAX; ++t) {              // the same trip count in every lane (shuffles)
        const bool on = act && t > s && t < T;
        float ck = 0.f, cq = 0.f;
        if (on) {
            const float* ga = g_lb + (size_t(t) * Hv + h) * D;
#pragma unroll
            for (int m = 0; m < NJ; ++m) {
                const int c = c8 + 8 * m;
                w[m] *= __ldg(ga + c);
                const float kw = ks[m] * w[m];
                ck = fmaf(kw, XP[t * D + c], ck);
                cq = fmaf(kw, XP[(TMAX + t) * D + c], cq);
            }
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            ck += __shfl_xor_sync(0xffffffffu, ck, o);
            cq += __shfl_xor_sync(0xffffffffu, cq, o);
        }
        if (c8 == 0 && on) {
            recj[t * RS + 4 + s] = ck;
            recj[t * RS + 4 + TMAX + s] = cq;
        }
    }
    named_bar(bar, 128);
}

template <typename IO, int TMAX, int G, bool COMMIT, bool TREE, bool GDK>
__global__ void __launch_bounds__(PipeCfg<IO, TMAX, G, COMMIT, TREE, GDK>::NTHR, 1)
gdn_verify_pipe_kernel(const VerifyArgs a, const __grid_constant__ CUtensorMap smap,
                       const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap cmap,
                       const __grid_constant__ CUtensorMap pmap, int n_units) {
    using Cfg = PipeCfg<IO, TMAX, G, COMMIT, TREE, GDK>;
    constexpr int D = Cfg::D, NP = Cfg::NP, XKB = Cfg::XKB, RS = Cfg::RS;
    constexpr int NXS = Cfg::NXS, NSS = Cfg::NSS;
    constexpr int NKS = Cfg::NKS, NTS = Cfg::NTS;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base, derived from the shared array itself so that every access stays
    // a shared-memory access for the compiler
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* kfull = bars;                      // K-block landed in its shared-memory slot
    uint64_t* kempty = kfull + NKS;              // slot free: read by the 4 convert warps, or
                                                 // (COMMIT) stored back by the store warp
    uint64_t* kconv = kempty + NKS;              // COMMIT: slot updated by the 4 convert warps
    uint64_t* tmfull = kconv + NKS;              // hi / lo of a K-block in its TMEM slot (4 warps)
    uint64_t* tmempty = tmfull + NTS;            // TMEM slot consumed by the MMAs (commit)
    uint64_t* tfull = tmempty + NTS;             // unit's P slot complete (commit)
    uint64_t* tempty = tfull + 2;                // unit's P slot read by the 4 epilogue warps
    uint64_t* sfull = tempty + 2;                // staged inputs landed
    uint64_t* sempty = sfull + 2;                // staging slot released by prep
    uint64_t* ufull = sempty + 2;                // unit prologue (records, meta) ready: epilogue
    uint64_t* uempty = ufull + 2;                // unit slot free: last MMA commit + 4 epilogue warps
    uint64_t* kpfull = uempty + 2;               // COMMIT: previous round's tape rows staged
    uint64_t* kpempty = kpfull + 2;              // COMMIT: commit slot read by convert and epilogue
    uint64_t* mdone = kpempty + 2;               // every MMA of this CTA complete
    uint64_t* winfull = mdone + 1;               // BIG: the unit's conv windows written (prep)
    uint64_t* vdone = mdone + 2;                 // BIG: v in TMEM, staged rows read (4 epilogue warps)
    uint64_t* xfull = mdone + 3;                 // unit's B tile written (prep): the MMAs may start,
                                                 // while prep goes on to the Gram block and records
    uint64_t* ebar = mdone + 5;                  // BIG: the epilogue's solve products complete (commit)
    uint64_t* edone = mdone + 6;                 // BIG: drain of the epilogue's products
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);
    float* scr = reinterpret_cast<float*>(smem + Cfg::OFF_SCR);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, Hk = a.Hk, Hv = a.Hv, C = a.C, W = a.W, B = a.B;
    // give-up time of the pipeline waits (the drains at the end keep the full limit)
    const uint64_t lim = a.wait_ns ? a.wait_ns : kWaitLimitNs;
    const int NR = COMMIT ? 2 * (W - 1) + T : W - 1 + T;
    const int n_my = blockIdx.x < n_units ? (n_units - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;

    if (tid == 0) {
        for (int i = 0; i < Cfg::NBAR; ++i) {
            uint64_t* bb = &bars[i];
            const bool four = (!COMMIT && bb >= kempty && bb < kempty + NKS) ||
                              (bb >= kconv && bb < kconv + NKS) || (bb >= tmfull && bb < tmfull + NTS) ||
                              (bb >= tempty && bb < tempty + 2) || bb == vdone;
            const bool kpe = bb >= kpempty && bb < kpempty + 2;
            mbar_init(bb, four ? 4 : kpe ? 8 : (bb >= uempty && bb < uempty + 2) ? 5 : 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tslot)), "r"(uint32_t(Cfg::TMEM_COLS)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tslot;

    auto unit_of = [&](int iu, int& l, int& b, int& kh) {
        const int u = blockIdx.x + iu * gridDim.x;
        kh = u % Hk;
        const int lbi = u / Hk;
        l = lbi / B;
        b = lbi - l * B;
    };
    // previous round's accepted count of sequence b (COMMIT); outside [0, T] it commits nothing
    // (the input loader reports it)
    auto n_prev = [&](int b) -> int {
        if (!COMMIT) return 0;
        const int n = __ldg(a.n_acc_prev + b);
        return (n < 0 || n > T) ? 0 : n;
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ state loader (whole warp)
        int s = 0, issued = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int iu = 0; iu < n_my && ok; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const size_t lb = size_t(l) * B + b;
            // K-block major, value heads minor: the order in which the MMAs consume them
            for (int kb = 0; kb < Cfg::KB && ok; ++kb) {
                for (int j = 0; j < G; ++j) {
                    const int row0 = int((lb * Hv + kh * G + j) * D);
                    if (!pwait_warp(&kempty[s], ph ^ 1, abort_flag, a.status, lim)) { ok = false; break; }
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&kfull[s], uint32_t(Cfg::KSLOT));
                        tma_load_2d(smem + Cfg::OFF_RING + size_t(s) * Cfg::KSLOT, &smap, kb * 32, row0,
                                    &kfull[s]);
                    }
                    __syncwarp();
                    ++issued;
                    if (++s == NKS) { s = 0; ph ^= 1; }
                }
            }
        }
        // drain: the copies in flight must land before the CTA may exit
        volatile int no_abort = 0;
        for (int k = 1; k <= NKS && k <= issued; ++k) {
            const int q = issued - k;
            pwait_warp(&kfull[q % NKS], uint32_t(q / NKS) & 1u, &no_abort, a.status);
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------------ input loader (whole warp)
        // staged layout per part: W-1 old conv-state rows, T qkv rows, (COMMIT) W-1 rows of the
        // previous round's qkv ending at row n-1; then the conv taps of every part [NPARTS][D][W].
        // All destinations are multiples of 128 bytes.
        const IO* cw = static_cast<const IO*>(a.conv_w);
        int issued = 0;
        // COMMIT: gate g'_s of lane (j, s) of a unit's previous round, loaded one unit ahead
        auto prev_gate = [&](int iu2) -> float {
            if (!COMMIT || iu2 >= n_my) return 1.f;
            int l2, b2, kh2;
            unit_of(iu2, l2, b2, kh2);
            const int n2 = n_prev(b2);
            const int gj = lane / TMAX, gs = lane - gj * TMAX;
            return (gj < G && gs < n2) ? __ldg(a.g_prev + ((size_t(l2) * B + b2) * T + gs) * Hv + kh2 * G + gj)
                                       : 1.f;
        };
        float gv_next = prev_gate(0);
        for (int iu = 0; iu < n_my; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const size_t lb = size_t(l) * B + b;
            const int ss = iu % NSS;
            IO* qs = reinterpret_cast<IO*>(smem + Cfg::OFF_STAGE + size_t(ss) * Cfg::STAGE_BYTES);
            IO* cws = qs + size_t(Cfg::NPARTS) * NR * D;
            int n = 0;
            const float gv = gv_next;
            if (COMMIT) {
                const int nr = __ldg(a.n_acc_prev + b);
                if ((nr < 0 || nr > T) && lane == 0 && kh == 0 && l == 0)
                    set_status(a.status, GDN_STATUS_BAD_NACC);
                n = n_prev(b);
                gv_next = prev_gate(iu + 1);
            }
            if (!pwait_warp(&sempty[ss], ((iu / NSS) & 1) ^ 1, abort_flag, a.status, lim)) break;
            if (lane == 0) {
                const int rows = (W - 1) + T + ((COMMIT && n > 0) ? W - 1 : 0);
                mbar_arrive_expect_tx(&sfull[ss], uint32_t(Cfg::NPARTS * (rows * D + D * W) * Cfg::ES));
#pragma unroll
                for (int part = 0; part < Cfg::NPARTS; ++part) {
                    const int cb = part == 0 ? kh * D
                                 : part == 1 ? Hk * D + kh * D : 2 * Hk * D + (kh * G + part - 2) * D;
                    IO* dst = qs + size_t(part) * NR * D;
                    if (W > 1) tma_load_2d(dst, &cmap, cb, int(lb * (W - 1)), &sfull[ss]);
                    tma_load_2d(dst + size_t(W - 1) * D, &qmap, cb, int(lb * T), &sfull[ss]);
                    if (COMMIT && n > 0 && W > 1)   // rows n-(W-1) .. n-1 (negative rows read as 0)
                        tma_load_2d(dst + size_t(W - 1 + T) * D, &pmap, cb, int(lb * T) + n - (W - 1),
                                    &sfull[ss]);
                    bulk_g2s(cws + size_t(part) * D * W, cw + (size_t(l) * C + cb) * W,
                             uint32_t(D * W * Cfg::ES), &sfull[ss]);
                }
            }
            __syncwarp();
            if (COMMIT) {
                // previous round's tape rows and gate coefficients of this unit
                const int ks = iu & 1;
                float* kp = reinterpret_cast<float*>(smem + Cfg::OFF_KP + size_t(ks) * Cfg::KP_BYTES);
                if (!pwait_warp(&kpempty[ks], ((iu >> 1) & 1) ^ 1, abort_flag, a.status, lim)) break;
                {
                    // c_s = Γ(s+1 .. n-1) and Γ(0 .. n-1) by a suffix-product scan over the lanes
                    // (lane j TMAX + s holds g'_s, 1 for s >= n): log2(TMAX) steps instead of a
                    // chain of TMAX shuffles
                    const int sj = lane / TMAX, ss2 = lane - sj * TMAX;
                    float x = gv;                    // becomes Π_{r = s .. TMAX-1} g'_r
#pragma unroll
                    for (int o = 1; o < TMAX; o <<= 1) {
                        const float y = __shfl_down_sync(0xffffffffu, x, o);
                        if (ss2 + o < TMAX) x *= y;
                    }
                    const float nx = __shfl_down_sync(0xffffffffu, x, 1);
                    const float cs = ss2 + 1 < TMAX ? nx : 1.f;
                    if (sj < G) {
                        if (ss2 < n) kp[Cfg::KP_C + sj * TMAX + ss2] = cs;
                        if (ss2 == 0) kp[Cfg::KP_GAM + sj] = x;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&kpfull[ks], uint32_t(n * (1 + G) * D * 4));
                    for (int s2 = 0; s2 < n; ++s2) {
                        bulk_g2s(kp + Cfg::KP_K + s2 * Cfg::KP_KS,
                                 a.tape_k_prev + ((lb * T + s2) * Hk + kh) * size_t(D), uint32_t(D * 4),
                                 &kpfull[ks]);
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            bulk_g2s(kp + Cfg::KP_DL + (j * TMAX + s2) * Cfg::KP_KS,
                                     a.tape_delta_prev + ((lb * T + s2) * Hv + kh * G + j) * size_t(D),
                                     uint32_t(D * 4), &kpfull[ks]);
                    }
                }
                __syncwarp();
            }
            ++issued;
        }
        volatile int no_abort = 0;
        for (int k = 1; k <= NSS && k <= issued; ++k) {
            const int q = issued - k;
            pwait_warp(&sfull[q % NSS], uint32_t(q / NSS) & 1u, &no_abort, a.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ mma (whole warp)
        // chain c of a unit slot: hi pass (N = 2NP) at c * CH_COLS, lo pass (N = NP) at + 2NP. Per
        // K-step the order is hi of every chain, then lo of every chain: the same accumulator comes
        // back only every 4 MMAs, past the tensor core's accumulate latency.
        constexpr int S = Cfg::S;
        constexpr uint32_t IDESC1 = umma_idesc_tf32(128, 2 * NP);
        constexpr uint32_t IDESC2 = umma_idesc_tf32(128, NP);
        const uint32_t sX0 = smem_u32(smem + Cfg::OFF_X);
        int ts = 0;
        uint32_t tph = 0;
        bool ok = true;
        for (int iu = 0; iu < n_my && ok; ++iu) {
            const int us = iu % NXS, ps = iu % Cfg::NUS;
            // the B tile alone is enough to start (the records are read by the epilogue warps only)
            if (!pwait_warp(&xfull[us], (iu / NXS) & 1, abort_flag, a.status, lim))
                break;
            if (!pwait_warp(&tempty[ps], ((iu / Cfg::NUS) & 1) ^ 1, abort_flag, a.status, lim)) break;
            const uint64_t db = umma_desc_sw128(sX0 + us * Cfg::NXT * Cfg::X_BYTES);
            const uint32_t dt = tbase + ps * Cfg::P_COLS;
            for (int kb = 0; kb < Cfg::KB; ++kb) {
                int slot[G];
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    if (!pwait_warp(&tmfull[ts], tph, abort_flag, a.status, lim)) ok = false;
                    slot[j] = ts;
                    if (++ts == NTS) { ts = 0; tph ^= 1; }
                }
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bk = db + uint64_t((kb * XKB + ks * 32) >> 4);
                    const uint32_t acc = (kb > 0 || ks >= S) ? 1u : 0u;
                    if constexpr (Cfg::BIG) {
                        // one NP-column accumulator per chain: S_hi·X_hi, S_hi·X_lo, S_lo·X_hi
                        const uint64_t bk_lo = bk + uint64_t((NP * 128) >> 4);
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            umma_tf32_ts_warp(dt + (j * S + ks % S) * Cfg::CH_COLS,
                                              tbase + Cfg::T_RING + slot[j] * 64 + ks * 8, bk, IDESC2, acc);
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            umma_tf32_ts_warp(dt + (j * S + ks % S) * Cfg::CH_COLS,
                                              tbase + Cfg::T_RING + slot[j] * 64 + ks * 8, bk_lo, IDESC2, 1u);
#pragma unroll
                        for (int j = 0; j < G; ++j)
                            umma_tf32_ts_warp(dt + (j * S + ks % S) * Cfg::CH_COLS,
                                              tbase + Cfg::T_RING + slot[j] * 64 + 32 + ks * 8, bk, IDESC2, 1u);
                    } else {
                        // GDK: head j reads its own B tile
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            const int c = j * S + ks % S;
                            const uint64_t bj = bk + uint64_t(((GDK ? j : 0) * Cfg::X_BYTES) >> 4);
                            umma_tf32_ts_warp(dt + c * Cfg::CH_COLS, tbase + Cfg::T_RING + slot[j] * 64 + ks * 8,
                                              bj, IDESC1, acc);
                        }
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            const int c = j * S + ks % S;
                            const uint64_t bj = bk + uint64_t(((GDK ? j : 0) * Cfg::X_BYTES) >> 4);
                            umma_tf32_ts_warp(dt + c * Cfg::CH_COLS + 2 * NP,
                                              tbase + Cfg::T_RING + slot[j] * 64 + 32 + ks * 8, bj, IDESC2, acc);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < G; ++j) umma_commit_warp(&tmempty[slot[j]]);
            }
            if (ok) {
                umma_commit_warp(&tfull[ps]);
                umma_commit_warp(&uempty[us]);
            }
        }
        // drain: every MMA must have completed before TMEM is released
        umma_commit_warp(mdone);
        volatile int no_abort = 0;
        pwait_warp(mdone, 0, &no_abort, a.status);
    } else if (warp < 6) {
        // ------------------------------------------------------------------ prep (128 threads)
        const int p = tid - 64, pw = warp - 2;
        const int gq = lane >> 2, gt4 = lane & 3;       // mma.sync fragment coordinates
        float* nrm = scr + Cfg::S_NRM;
        float* inv = scr + Cfg::S_INV;
        float* gp = scr + Cfg::S_GP;
        float* gram = scr + Cfg::S_GRAM;
        for (int iu = 0; iu < n_my; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const size_t lb = size_t(l) * B + b;
            const int ss = iu % NSS, us = iu % NXS;
            unsigned char* st = smem + Cfg::OFF_STAGE + size_t(ss) * Cfg::STAGE_BYTES;
            const IO* qs = reinterpret_cast<const IO*>(st);
            const IO* cws = qs + size_t(Cfg::NPARTS) * NR * D;
            unsigned char* Xb = smem + Cfg::OFF_X + size_t(us) * Cfg::NXT * Cfg::X_BYTES;
            float* meta = reinterpret_cast<float*>(smem + Cfg::OFF_META + size_t(us) * Cfg::META_BYTES);
            // gates of this thread's (value head gj, position gt), loaded early; with one decay per
            // key channel the record's γ is 1 and the thread loads its channel p of every gate row
            float g_in = GDK ? 1.f : 0.f, b_in = 0.f;
            const int gj = p / TMAX, gt = p - gj * TMAX;
            if (p < G * TMAX && gt < T) {
                if constexpr (!GDK) g_in = __ldg(a.g + (lb * T + gt) * Hv + kh * G + gj);
                b_in = __ldg(a.beta + (lb * T + gt) * Hv + kh * G + gj);
            }
            float gch[GDK ? TMAX : 1][GDK ? G : 1];
            if constexpr (GDK) {
#pragma unroll
                for (int t = 0; t < TMAX; ++t)
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        gch[t][j] = t < T ? __ldg(a.g + ((lb * T + t) * Hv + kh * G + j) * size_t(D) + p) : 1.f;
            }
            // conv window row r (0 .. W-2): old conv-state row r + n, or (COMMIT, r + n ≥ W-1) the
            // previous round's raw row staged at W-1+T+r
            const int n = n_prev(b);
            int* par_s = reinterpret_cast<int*>(scr + Cfg::S_PAR);
            int* win_s = reinterpret_cast<int*>(scr + Cfg::S_WIN);
            if constexpr (TREE) {
                // parents (a bad tree reports GDN_STATUS_BAD_PARENT and runs as a chain) and each
                // node's conv window: itself, its nearest ancestors, then the conv state's rows
                int* bad = win_s + 4 * TMAX;
                const int pv = p < T ? __ldg(a.parent + size_t(b) * T + p) : 0;
                if (p == 0) *bad = 0;
                named_bar(1, 128);
                if (p < T && (pv < -1 || pv >= p)) atomicOr(bad, 1);
                named_bar(1, 128);
                const int isbad = *bad;
                if (p < T) par_s[p] = isbad ? p - 1 : pv;
                if (isbad && p == 0) set_status(a.status, GDN_STATUS_BAD_PARENT);
                named_bar(1, 128);
                // stored as element offsets of the staged rows; taps d >= W (weight 0) and nodes
                // past T point at a valid row (the node's own, or row 0)
                if (p < TMAX) {
                    int x = p < T ? p : -1, e = 0;
#pragma unroll
                    for (int d = 0; d < 4; ++d) {
                        int src = p < T ? W - 1 + p : 0;
                        if (d < W && p < T) {
                            if (x >= 0) { src = W - 1 + x; x = par_s[x]; }
                            else { src = W - 2 - e; ++e; }
                        }
                        win_s[p * 4 + d] = src * D;
                    }
                }
                if constexpr (Cfg::BIG) {
                    named_bar(1, 128);
                    if (p == 0) mbar_arrive(winfull);      // the epilogue warps' v conv may start
                }
            }
            pwait(&sfull[ss], (iu / NSS) & 1, abort_flag, a.status, lim);
            if constexpr (Cfg::BIG) {
                // one meta slot: the B tile is free once the previous unit's products are done;
                // its records are waited for just before this unit's are written (below)
                if (iu > 0) pwait(&tfull[(iu - 1) % Cfg::NUS], uint32_t((iu - 1) / Cfg::NUS) & 1u, abort_flag, a.status, lim);
            } else {
                pwait(&uempty[us], ((iu / NXS) & 1) ^ 1, abort_flag, a.status, lim);
            }
            if constexpr (TREE) {
                named_bar(1, 128);      // windows written
                // conv + SiLU over each node's window. Trees of 32 nodes: the prep warps take q and
                // k (one part and two channels per thread), the epilogue warps the v heads (into
                // TMEM). Smaller trees: thread p takes channels 2 (p mod 64) + {0, 1} of parts
                // 2 (p / 64) + {0, 1}.
                if constexpr (Cfg::BIG) {
                    tree_conv_parts<Cfg, 1, true>(p >> 6, 2 * (p & 63), qs, cws, NR, W, T, win_s, Xb, meta);
                } else {
                    if (p < 64)
                        tree_conv_parts<Cfg, 2, true>(0, 2 * p, qs, cws, NR, W, T, win_s, Xb, meta);
                    else
                        tree_conv_parts<Cfg, G, false>(2, 2 * (p - 64), qs, cws, NR, W, T, win_s, Xb, meta);
                }
                named_bar(1, 128);
                if (!Cfg::BIG && p == 0) mbar_arrive(&sempty[ss]);     // every staged row has been read
                // norms: warp pw takes rows pw, pw + 4, ..; lane = 4 channels (one 16-byte chunk).
                // The tape keeps the normalised k; the B tile stays raw (the coefficients and the
                // epilogue apply the inverse norms).
                {
                    constexpr int RPW = 2 * TMAX / 4;          // rows per warp (a power of 2)
                    float sq[RPW];
#pragma unroll
                    for (int m = 0; m < RPW; ++m) {
                        const float4 x = *reinterpret_cast<const float4*>(Xb + sw128_off(pw + 4 * m, 4 * lane, XKB));
                        sq[m] = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                    }
                    int ix;                                    // row pw + 4 ix, held by lanes ix * 32 / RPW ..
                    const float iv = inv_sqrt_nr(warp_sum_many<RPW>(sq, lane, &ix) + a.l2_eps);
                    inv[pw + 4 * ix] = iv;                     // lanes sharing ix write the same value
#pragma unroll
                    for (int m = 0; m < TMAX / 4; ++m) {       // k rows: pw + 4 m < TMAX
                        const int r = pw + 4 * m;
                        const float ivm = __shfl_sync(0xffffffffu, iv, m * (32 / RPW));
                        const float4 x = *reinterpret_cast<const float4*>(Xb + sw128_off(r, 4 * lane, XKB));
                        st_global_if(a.tape_k + ((lb * T + r) * Hk + kh) * size_t(D) + 4 * lane,
                                     make_float4(x.x * ivm, x.y * ivm, x.z * ivm, x.w * ivm), r < T);
                    }
                }
#pragma unroll
                for (int n2 = 2 * TMAX; n2 < NP; ++n2) {
                    *reinterpret_cast<float*>(Xb + sw128_off(n2, p, XKB)) = 0.f;
                    *reinterpret_cast<float*>(Xb + sw128_off(NP + n2, p, XKB)) = 0.f;
                }
                if (!Cfg::BIG && p < G * TMAX) {
                    float* rec = meta + Cfg::M_REC + p * RS;
                    rec[1] = g_in;
                    rec[2] = b_in;
                }
            } else {
            // conv + SiLU of channel p of every part (one loop body for all parts keeps the code
            // small: q and k stay in registers, each v goes to the meta slot)
            float yq[TMAX], yk[TMAX];
#pragma unroll 1
            for (int part = 0; part < Cfg::NPARTS; ++part) {
                const IO* col = qs + size_t(part) * NR * D + p;
                const IO* wp = cws + (size_t(part) * D + p) * W;
                float wr[4];     // wr[d] multiplies the row at distance d (0 = current token)
                if (W == 4) {
                    const uint2 w4 = *reinterpret_cast<const uint2*>(wp);
                    const IO* wv = reinterpret_cast<const IO*>(&w4);
#pragma unroll
                    for (int d = 0; d < 4; ++d) wr[d] = io_to_f(wv[3 - d]);
                } else {
#pragma unroll
                    for (int d = 0; d < 4; ++d) wr[d] = (d < W) ? io_to_f(wp[W - 1 - d]) : 0.f;
                }
                float E[3 + TMAX];
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int r = k + W - 4;
                    const int src = r + n < W - 1 ? r + n : W - 1 + T + r;
                    E[k] = (r >= 0) ? io_to_f(col[size_t(src) * D]) : 0.f;
                }
#pragma unroll
                for (int t = 0; t < TMAX; ++t) E[3 + t] = (t < T) ? io_to_f(col[size_t(W - 1 + t) * D]) : 0.f;
                if (COMMIT && n > 0) {
                    // the committed window is the new conv state: row r is E[r + 4 - W] (exact
                    // copies), stashed for the epilogue warps to write out
                    IO* cw_s = reinterpret_cast<IO*>(meta + Cfg::M_CW) + size_t(part) * 3 * D + p;
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const int r = k + W - 4;
                        if (r >= 0) IoTraits<IO>::store(cw_s, size_t(r) * D, E[k]);
                    }
                }
                float yv[TMAX];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    float acc = wr[3] * E[t];
                    acc = fmaf(wr[2], E[t + 1], acc);
                    acc = fmaf(wr[1], E[t + 2], acc);
                    acc = fmaf(wr[0], E[t + 3], acc);
                    yv[t] = (t < T) ? silu_fast(acc) : 0.f;
                }
                if (part == 0) {
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) yq[t] = yv[t];
                } else if (part == 1) {
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) yk[t] = yv[t];
                } else {
#pragma unroll
                    for (int t = 0; t < TMAX; ++t) meta[Cfg::M_V + ((part - 2) * TMAX + t) * D + p] = yv[t];
                }
            }
            // norms of k_t (columns 0..TMAX-1) and q_t (columns TMAX..2TMAX-1)
            {
                float sq[2 * TMAX];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    sq[t] = yk[t] * yk[t];
                    sq[TMAX + t] = yq[t] * yq[t];
                }
                int ix;
                const float s = warp_sum_many<2 * TMAX>(sq, lane, &ix);
                if ((lane & (32 / (2 * TMAX) - 1)) == 0) nrm[pw * 2 * TMAX + ix] = s;
            }
            named_bar(1, 128);
            if (p == 0) mbar_arrive(&sempty[ss]);         // every staged row has been read
            if (p < 2 * TMAX)
                inv[p] = 1.0f / sqrtf(nrm[p] + nrm[2 * TMAX + p] + nrm[4 * TMAX + p] +
                                      nrm[6 * TMAX + p] + a.l2_eps);
            named_bar(1, 128);
            // B tile rows n < NP: X as raw fp32 (the tensor core reads it as X_hi = trunc_tf32(X));
            // rows NP + n: X_lo = X − X_hi. Also the tape k, v values, gates. GDK: tile j holds
            // A_t ⊙ k_t and A_t ⊙ q_t with head j's running product A_t of channel p's gates, and
            // the plain rows go to the meta slot for the epilogue's Gram.
            if constexpr (GDK) {
                float cum[G];
#pragma unroll
                for (int j = 0; j < G; ++j) cum[j] = 1.f;
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    const float kn = yk[t] * inv[t], qn = yq[t] * inv[TMAX + t];
                    meta[Cfg::M_XP + t * D + p] = kn;
                    meta[Cfg::M_XP + (TMAX + t) * D + p] = qn;
                    st_global_if(a.tape_k + ((lb * T + t) * Hk + kh) * size_t(D) + p, kn, t < T);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        cum[j] *= gch[t][j];
                        unsigned char* Xj = Xb + size_t(j) * Cfg::X_BYTES;
                        const float xk = kn * cum[j], xq = qn * cum[j];
                        *reinterpret_cast<float*>(Xj + sw128_off(t, p, XKB)) = xk;
                        *reinterpret_cast<float*>(Xj + sw128_off(NP + t, p, XKB)) = xk - tf32_trunc(xk);
                        *reinterpret_cast<float*>(Xj + sw128_off(TMAX + t, p, XKB)) = xq;
                        *reinterpret_cast<float*>(Xj + sw128_off(NP + TMAX + t, p, XKB)) = xq - tf32_trunc(xq);
                    }
                }
            } else {
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                const float kn = yk[t] * inv[t], qn = yq[t] * inv[TMAX + t];
                *reinterpret_cast<float*>(Xb + sw128_off(t, p, XKB)) = kn;
                *reinterpret_cast<float*>(Xb + sw128_off(NP + t, p, XKB)) = kn - tf32_trunc(kn);
                *reinterpret_cast<float*>(Xb + sw128_off(TMAX + t, p, XKB)) = qn;
                *reinterpret_cast<float*>(Xb + sw128_off(NP + TMAX + t, p, XKB)) = qn - tf32_trunc(qn);
                st_global_if(a.tape_k + ((lb * T + t) * Hk + kh) * size_t(D) + p, kn, t < T);
            }
            }
#pragma unroll
            for (int j = 0; j < Cfg::NXT; ++j) {
                unsigned char* Xj = Xb + size_t(j) * Cfg::X_BYTES;
#pragma unroll
                for (int n2 = 2 * TMAX; n2 < NP; ++n2) {
                    *reinterpret_cast<float*>(Xj + sw128_off(n2, p, XKB)) = 0.f;
                    *reinterpret_cast<float*>(Xj + sw128_off(NP + n2, p, XKB)) = 0.f;
                }
            }
            if (p < G * TMAX) {
                float* rec = meta + Cfg::M_REC + p * RS;      // record (gj, gt)
                rec[1] = g_in;
                rec[2] = b_in;
            }
            }   // chain
            fence_async_smem();
            named_bar(1, 128);
            if (p == 0) mbar_arrive(&xfull[us]);   // the B tile is complete: the MMAs may start
            // BIG: the Gram block lives in the meta slot
            if constexpr (Cfg::BIG) gram = meta + Cfg::M_V;
            if constexpr ((TREE || TMAX < 16) && !GDK) {   // 16-position chains and GDK: the epilogue warps
            // Gram block on the warp tensor path: D[m][n] = X_m · k_n, 3xTF32 (hi·hi + hi·lo + lo·hi);
            // rows m: k_0.., q_0.. (zero beyond 2 TMAX). One 16 x 8 tile: each warp takes 32 channels
            // and the partials are summed; four tiles (TMAX = 16): warp pw takes tile pw, all channels.
            if constexpr (Cfg::GRAM_TILES >= 4) {
              // a warp's tiles (one, or four sharing the column block k_{8 pw ..}) in one pass over
              // the channels, hi·hi + lo·hi and hi·lo in separate accumulators: 2 TPW independent
              // chains
              constexpr int NTN = (TMAX + 7) / 8, TPW = Cfg::GRAM_TILES / 4;
              static_assert(TPW == 1 || NTN == 4, "a warp's tiles share their column block");
              const int nt = pw % NTN;
              // one tile per warp: four accumulator sets, rotated over the K-steps
              constexpr int NACC = TPW == 1 ? 4 : 1, KUNROLL = TPW == 1 ? 4 : 2;
              float acc[TPW * NACC][4], acl[TPW * NACC][4];
#pragma unroll
              for (int m = 0; m < TPW * NACC; ++m)
#pragma unroll
                  for (int e = 0; e < 4; ++e) { acc[m][e] = 0.f; acl[m][e] = 0.f; }
#pragma unroll (KUNROLL)
              for (int ks = 0; ks < 16; ++ks) {
                const int ka = NACC == 1 ? 0 : (ks & 3);
                // B: rows 8 nt .., channels 8 ks + 0..3 and + 4..7 (ldmatrix, lanes 0..15)
                uint32_t rb[2];
                ldsm_x2(smem_u32(Xb + sw128_off(8 * nt + (lane & 7), 8 * ks + ((lane >> 3) & 1) * 4, XKB)), rb);
                const float bv0 = __uint_as_float(rb[0]), bv1 = __uint_as_float(rb[1]);
                const float bh0 = tf32_trunc(bv0), bh1 = tf32_trunc(bv1);
                const uint32_t bl0 = __float_as_uint(tf32_trunc(bv0 - bh0));
                const uint32_t bl1 = __float_as_uint(tf32_trunc(bv1 - bh1));
                uint32_t ahi[TPW][4], alo[TPW][4];
#pragma unroll
                for (int m = 0; m < TPW; ++m) {
                    const int mt = TPW == 1 ? pw / NTN : m;
                    // A: rows 16 mt + 0..7 / 8..15, channels 8 ks + 0..3 / 4..7 (ldmatrix)
                    uint32_t ra[4];
                    ldsm_x4(smem_u32(Xb + sw128_off(16 * mt + ((lane >> 3) & 1) * 8 + (lane & 7),
                                                    8 * ks + (lane >> 4) * 4, XKB)), ra);
                    const float av[4] = {__uint_as_float(ra[0]), __uint_as_float(ra[1]), __uint_as_float(ra[2]),
                                         __uint_as_float(ra[3])};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float h = tf32_trunc(av[e]);
                        ahi[m][e] = __float_as_uint(h);
                        alo[m][e] = __float_as_uint(tf32_trunc(av[e] - h));
                    }
                }
#pragma unroll
                for (int m = 0; m < TPW; ++m) {
                    mma_tf32_16x8x8(acc[m + ka], ahi[m], __float_as_uint(bh0), __float_as_uint(bh1));
                    mma_tf32_16x8x8(acl[m + ka], ahi[m], bl0, bl1);
                }
#pragma unroll
                for (int m = 0; m < TPW; ++m)
                    mma_tf32_16x8x8(acc[m + ka], alo[m], __float_as_uint(bh0), __float_as_uint(bh1));
              }
#pragma unroll
              for (int q2 = 1; q2 < NACC; ++q2)
#pragma unroll
                  for (int e = 0; e < 4; ++e) { acc[0][e] += acc[q2][e]; acl[0][e] += acl[q2][e]; }
              // Gr[a][c] = k_a · X_c = D[c][a]
#pragma unroll
              for (int m = 0; m < TPW; ++m) {
                const int mt = TPW == 1 ? pw / NTN : m;
                const int c0 = 16 * mt + gq, a0 = 8 * nt + 2 * gt4;
                gram[a0 * 2 * TMAX + c0] = acc[m][0] + acl[m][0];
                gram[(a0 + 1) * 2 * TMAX + c0] = acc[m][1] + acl[m][1];
                gram[a0 * 2 * TMAX + c0 + 8] = acc[m][2] + acl[m][2];
                gram[(a0 + 1) * 2 * TMAX + c0 + 8] = acc[m][3] + acl[m][3];
              }
            } else {
              {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const int ch = 32 * pw + 8 * ks + gt4;
                    float av[4];
                    av[0] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch, XKB));
                    av[2] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch + 4, XKB));
                    av[1] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch, XKB)) : 0.f;
                    av[3] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch + 4, XKB)) : 0.f;
                    const float bv0 = gq < TMAX ? av[0] : 0.f, bv1 = gq < TMAX ? av[2] : 0.f;
                    uint32_t ahi[4], alo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float h = tf32_trunc(av[e]);
                        ahi[e] = __float_as_uint(h);
                        alo[e] = __float_as_uint(tf32_trunc(av[e] - h));
                    }
                    const float bh0 = tf32_trunc(bv0), bh1 = tf32_trunc(bv1);
                    const uint32_t bl0 = __float_as_uint(tf32_trunc(bv0 - bh0));
                    const uint32_t bl1 = __float_as_uint(tf32_trunc(bv1 - bh1));
                    mma_tf32_16x8x8(acc, ahi, __float_as_uint(bh0), __float_as_uint(bh1));
                    mma_tf32_16x8x8(acc, ahi, bl0, bl1);
                    mma_tf32_16x8x8(acc, alo, __float_as_uint(bh0), __float_as_uint(bh1));
                }
                float* g4 = gp + pw * 128;
                g4[gq * 8 + 2 * gt4] = acc[0];
                g4[gq * 8 + 2 * gt4 + 1] = acc[1];
                g4[(gq + 8) * 8 + 2 * gt4] = acc[2];
                g4[(gq + 8) * 8 + 2 * gt4 + 1] = acc[3];
              }
              named_bar(1, 128);
              {
                const int m = p >> 3, nn = p & 7;
                if (m < 2 * TMAX && nn < TMAX)
                    gram[nn * 2 * TMAX + m] = gp[p] + gp[128 + p] + gp[256 + p] + gp[384 + p];
              }
            }
            named_bar(1, 128);
            if constexpr (TREE) {
                // per (value head, node v): walk v's ancestors x (nearest first). CK[v][x] =
                // Γ(x→v) k_x·k_v and CQ[v][x] = Γ(x→v) k_x·q_v, with Γ(x→v) the gates of the
                // ancestors strictly between x and v; zero for every other x. c0 = every
                // ancestor's gate. The Gram block is raw: the inverse norms are applied here.
                if constexpr (Cfg::BIG) {
                    // the previous unit's epilogue has read its records
                    pwait(&uempty[us], ((iu / NXS) & 1) ^ 1, abort_flag, a.status, lim);
                    if (p < G * TMAX) {
                        meta[Cfg::M_FLD + gj * Cfg::FJ + Cfg::F_GAM + gt] = g_in;
                        meta[Cfg::M_FLD + gj * Cfg::FJ + Cfg::F_BET + gt] = b_in;
                    }
                    if (p < TMAX) reinterpret_cast<int*>(meta + Cfg::M_PAR)[p] = p < T ? par_s[p] : -1;
                    constexpr int NZ = 2 * TMAX * TMAX / 4;          // CK, CQ of one head in float4
#pragma unroll 1
                    for (int z = p; z < G * NZ; z += 128) {
                        const int zj = z / NZ;
                        reinterpret_cast<float4*>(meta + Cfg::M_REC + zj * Cfg::RJ + Cfg::F_CKT)[z - zj * NZ] =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    named_bar(1, 128);
                    for (int idx = p; idx < G * TMAX; idx += 128) {
                        const int fj = idx / TMAX, fv = idx - fj * TMAX;
                        if (fv >= T) continue;
                        float* hb = meta + Cfg::M_REC + fj * Cfg::RJ;
                        float* fb = meta + Cfg::M_FLD + fj * Cfg::FJ;
                        const float ik = inv[fv], iq = inv[TMAX + fv];
                        float coef = 1.f;
                        int y = par_s[fv];
                        while (y >= 0) {
                            const float iy = inv[y] * coef;
                            hb[Cfg::F_CKT + y * TMAX + fv] = iy * ik * gram[y * 2 * TMAX + fv];
                            hb[Cfg::F_CQT + y * TMAX + fv] = iy * iq * gram[y * 2 * TMAX + TMAX + fv];
                            coef *= fb[Cfg::F_GAM + y];
                            y = par_s[y];
                        }
                        fb[Cfg::F_C0K + fv] = coef * ik;
                        fb[Cfg::F_C0Q + fv] = coef * iq;
                        fb[Cfg::F_KQ + fv] = gram[fv * 2 * TMAX + TMAX + fv] * ik * iq;
                    }
                } else
                for (int idx = p; idx < G * TMAX; idx += 128) {
                    const int fj = idx / TMAX, fv = idx - fj * TMAX;
                    if (fv < T) {
                        const float* hrec = meta + Cfg::M_REC + fj * TMAX * RS;     // γ at [y * RS + 1]
                        float* rec = meta + Cfg::M_REC + idx * RS;
                        float4* cz = reinterpret_cast<float4*>(rec + Cfg::HDR);
#pragma unroll
                        for (int z = 0; z < 2 * TMAX / 4; ++z) cz[z] = make_float4(0.f, 0.f, 0.f, 0.f);
                        const float ik = inv[fv], iq = inv[TMAX + fv];
                        float coef = 1.f;
                        unsigned gmask = 0;
                        int y = par_s[fv];
                        while (y >= 0) {
                            const float iy = inv[y] * coef;
                            rec[Cfg::HDR + y] = iy * ik * gram[y * 2 * TMAX + fv];
                            rec[Cfg::HDR + TMAX + y] = iy * iq * gram[y * 2 * TMAX + TMAX + fv];
                            gmask |= 1u << (y >> 2);
                            coef *= hrec[y * RS + 1];
                            y = par_s[y];
                        }
                        rec[0] = coef * ik;
                        rec[3] = gram[fv * 2 * TMAX + TMAX + fv] * ik * iq;
                        rec[4] = coef * iq;
                        rec[5] = __uint_as_float(gmask);
                    }
                }
            } else {
            if constexpr (TMAX >= 16) {
            // per (value head, position v), walking back over x = v-1 .. 0: CK[v][x] =
            // Γ(x+1..v-1) k_x·k_v and CQ[v][x] = Γ(x+1..v-1) k_x·q_v; c0[v] = Γ(0..v-1), k_v·q_v
            for (int idx = p; idx < G * TMAX; idx += 128) {
                const int fj = idx / TMAX, fv = idx - fj * TMAX;
                if (fv < T) {
                    const float* hrec = meta + Cfg::M_REC + fj * TMAX * RS;     // γ at [y * RS + 1]
                    float* rec = meta + Cfg::M_REC + idx * RS;
                    float coef = 1.f;
                    for (int fx = fv - 1; fx >= 0; --fx) {
                        rec[4 + fx] = coef * gram[fx * 2 * TMAX + fv];
                        rec[4 + TMAX + fx] = coef * gram[fx * 2 * TMAX + TMAX + fv];
                        coef *= hrec[fx * RS + 1];
                    }
                    rec[0] = coef;
                    rec[3] = gram[fv * 2 * TMAX + TMAX + fv];
                }
            }
            } else {
            // per value head, one thread per (v, x ≤ v): CK[v][x] = Γ(x→v-1) k_x·k_v and
            // CQ[v][x] = Γ(x→v-1) k_x·q_v for x < v; c0[v] = Γ(root→v-1) and k_v·q_v for x = v
            for (int idx = p; idx < G * TMAX * TMAX; idx += 128) {
                const int fj = idx / (TMAX * TMAX), fv = (idx / TMAX) % TMAX, fx = idx % TMAX;
                if (fv < T && fx <= fv) {
                    const float* hrec = meta + Cfg::M_REC + fj * TMAX * RS;     // γ at [y * RS + 1]
                    float* rec = meta + Cfg::M_REC + (fj * TMAX + fv) * RS;
                    const int y0 = fx < fv ? fx + 1 : 0;
                    float coef = 1.f;
#pragma unroll
                    for (int yy = 0; yy < TMAX - 1; ++yy)
                        if (yy >= y0 && yy < fv) coef *= hrec[yy * RS + 1];
                    if (fx < fv) {
                        rec[4 + fx] = coef * gram[fx * 2 * TMAX + fv];
                        rec[4 + TMAX + fx] = coef * gram[fx * 2 * TMAX + TMAX + fv];
                    } else {
                        rec[0] = coef;
                        rec[3] = gram[fv * 2 * TMAX + TMAX + fv];
                    }
                }
            }
            }
            }
            }
            named_bar(1, 128);
            if (p == 0) mbar_arrive(&ufull[us]);
            if constexpr (Cfg::BIG) {
                // staged rows and windows stay until the epilogue warps' v conv has read them
                pwait(vdone, uint32_t(iu & 1), abort_flag, a.status, lim);
                if (p == 0) mbar_arrive(&sempty[ss]);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------------ convert (128 threads)
        // thread = state row: S_hi and S_lo of its 32 columns of each K-block into the TMEM ring (two
        // halves of 16). COMMIT, n > 0: then S_n = Γ S_0 + A K'ᵀ for the warp's 32 rows of the K-block
        // with mma.sync and written back in place for the store warp. Fragment row m of a 16-row
        // tile maps to state row 8 (m / 8) + 2 (m mod 4) + (m / 4 mod 2): each half-warp then touches
        // rows with distinct (row mod 8) / 2, so its 8-byte accesses in the 128-byte-swizzled tile
        // are free of bank conflicts.
        const int q4 = warp & 3, row = 32 * q4 + lane;
        const int gq = lane >> 2, gt4 = lane & 3;
        const int prow = 2 * (gq & 3) + (gq >> 2);        // fragment row gq (and gq + 8) -> tile row
        int s = 0, ts = 0;
        uint32_t ph = 0, tph = 0;
        for (int iu = 0; iu < n_my; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const int n = n_prev(b);
            const float* kp = reinterpret_cast<const float*>(smem + Cfg::OFF_KP + size_t(iu & 1) * Cfg::KP_BYTES);
            if (COMMIT) pwait(&kpfull[iu & 1], (iu >> 1) & 1, abort_flag, a.status, lim);
            for (int kb = 0; kb < Cfg::KB; ++kb) {
#pragma unroll 1
                for (int j = 0; j < G; ++j) {
                    pwait(&kfull[s], ph, abort_flag, a.status, lim);
                    pwait(&tmempty[ts], tph ^ 1, abort_flag, a.status, lim);
                    tc_fence_after();
                    unsigned char* Ab = smem + Cfg::OFF_RING + size_t(s) * Cfg::KSLOT;
                    const unsigned char* At = Ab + row * 128;
                    const uint32_t ta = tbase + Cfg::T_RING + ts * 64 + (uint32_t(32 * q4) << 16);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const float4 x = *reinterpret_cast<const float4*>(At + (((4 * hh + c) ^ (row & 7)) << 4));
                            const float v4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float h = tf32_trunc(v4[e]);
                                hi[4 * c + e] = __float_as_uint(h);
                                lo[4 * c + e] = __float_as_uint(v4[e] - h);
                            }
                        }
                        tmem_st16(ta + hh * 16, hi);
                        tmem_st16(ta + 32 + hh * 16, lo);
                    }
                    if (!COMMIT) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&kempty[s]);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tmfull[ts]);
                    if (COMMIT) {
                        if (n > 0) {
                            // A fragments (m16n8k8: a0 (r, s), a1 (r + 8, s), a2 (r, s + 4),
                            // a3 (r + 8, s + 4), r = r0 + gq, s = gt4) of A[i][s] = c_s δ_s[i],
                            // zero for s ≥ n; two 16-row tiles
                            uint32_t afh[2][4], afl[2][4];
                            const float gm = kp[Cfg::KP_GAM + j];
#pragma unroll
                            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int r = 32 * q4 + 16 * rt + prow + ((e & 1) ? 8 : 0);
                                    const int s2 = gt4 + ((e & 2) ? 4 : 0);
                                    const float av = s2 < n ? kp[Cfg::KP_C + j * TMAX + s2] *
                                                                  kp[Cfg::KP_DL + (j * TMAX + s2) * Cfg::KP_KS + r]
                                                            : 0.f;
                                    const float h = tf32_trunc(av);
                                    afh[rt][e] = __float_as_uint(h);
                                    afl[rt][e] = __float_as_uint(tf32_trunc(av - h));
                                }
#pragma unroll
                            for (int ct = 0; ct < 4; ++ct) {
                                // B'[k][col] = k'_k[kb * 32 + 8 ct + col]: b0 (k = gt4), b1 (k = gt4 + 4)
                                const int cc = kb * 32 + 8 * ct + gq;
                                const float kv0 = gt4 < n ? kp[Cfg::KP_K + gt4 * Cfg::KP_KS + cc] : 0.f;
                                const float kv1 = gt4 + 4 < n ? kp[Cfg::KP_K + (gt4 + 4) * Cfg::KP_KS + cc] : 0.f;
                                const float kb0 = tf32_trunc(kv0), kb1 = tf32_trunc(kv1);
                                const uint32_t bh0 = __float_as_uint(kb0), bh1 = __float_as_uint(kb1);
                                const uint32_t bl0 = __float_as_uint(tf32_trunc(kv0 - kb0));
                                const uint32_t bl1 = __float_as_uint(tf32_trunc(kv1 - kb1));
#pragma unroll
                                for (int rt = 0; rt < 2; ++rt) {
                                    float u[4] = {0.f, 0.f, 0.f, 0.f};
                                    mma_tf32_16x8x8(u, afh[rt], bh0, bh1);
                                    mma_tf32_16x8x8(u, afh[rt], bl0, bl1);
                                    mma_tf32_16x8x8(u, afl[rt], bh0, bh1);
                                    // u: (r, c), (r, c + 1), (r + 8, c), (r + 8, c + 1), c = 8 ct + 2 gt4
#pragma unroll
                                    for (int hr = 0; hr < 2; ++hr) {
                                        const int r = 32 * q4 + 16 * rt + prow + 8 * hr;
                                        const int c = 8 * ct + 2 * gt4;
                                        float2* pp = reinterpret_cast<float2*>(
                                            Ab + r * 128 + ((((c >> 2) ^ (r & 7))) << 4) + (c & 3) * 4);
                                        const float2 old = *pp;
                                        *pp = make_float2(fmaf(gm, old.x, u[2 * hr]),
                                                          fmaf(gm, old.y, u[2 * hr + 1]));
                                    }
                                }
                            }
                            fence_async_smem();   // the store warp's TMA reads the update
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&kconv[s]);
                    }
                    if (++s == NKS) { s = 0; ph ^= 1; }
                    if (++ts == NTS) { ts = 0; tph ^= 1; }
                }
            }
            if (COMMIT) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&kpempty[iu & 1]);
            }
        }
    } else if (COMMIT && warp == 15) {
        // ------------------------------------------------------------------ store (whole warp)
        // committed K-blocks back to the state by TMA store (lane 0: its bulk groups); a slot is
        // freed as soon as its store has read it (keeping stores in flight longer holds slots the
        // loader needs and measured slower)
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int iu = 0; iu < n_my && ok; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const size_t lb = size_t(l) * B + b;
            const int n = n_prev(b);
            for (int kb = 0; kb < Cfg::KB && ok; ++kb) {
                for (int j = 0; j < G; ++j) {
                    if (!pwait_warp(&kconv[s], ph, abort_flag, a.status, lim)) { ok = false; break; }
                    if (n > 0 && lane == 0) {
                        tma_store_2d(&smap, smem + Cfg::OFF_RING + size_t(s) * Cfg::KSLOT, kb * 32,
                                     int((lb * Hv + kh * G + j) * D));
                        bulk_commit();
                        bulk_wait_read_all();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&kempty[s]);
                    if (++s == NKS) { s = 0; ph ^= 1; }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if (warp >= 10 && warp < 14) {
        // ------------------------------------------------------------------ epilogue (128 threads)
        const int q4 = warp & 3, i = 32 * q4 + lane;
        IO* out = static_cast<IO*>(a.out);
        const float scale = a.qk_scale;
        constexpr int S = Cfg::S;
        for (int iu = 0; iu < n_my; ++iu) {
            int l, b, kh;
            unit_of(iu, l, b, kh);
            const size_t lb = size_t(l) * B + b;
            const int us = iu % NXS;
            const float* meta = reinterpret_cast<const float*>(smem + Cfg::OFF_META + size_t(us) * Cfg::META_BYTES);
            const int n = n_prev(b);
            const float* kp = reinterpret_cast<const float*>(smem + Cfg::OFF_KP + size_t(iu & 1) * Cfg::KP_BYTES);
            if constexpr (Cfg::BIG) {
                // the v heads of this unit's tree conv, into TMEM (the prep warps take q and k); the
                // previous unit's epilogue, just finished by these warps, has read the old v
                const IO* qs = reinterpret_cast<const IO*>(smem + Cfg::OFF_STAGE + size_t(iu % NSS) * Cfg::STAGE_BYTES);
                pwait(winfull, uint32_t(iu & 1), abort_flag, a.status, lim);
                pwait(&sfull[iu % NSS], uint32_t(iu / NSS) & 1u, abort_flag, a.status, lim);
                tc_fence_after();
                tree_vconv_tmem<Cfg>(i, qs, qs + size_t(Cfg::NPARTS) * NR * D, NR, W, T,
                                     reinterpret_cast<const int*>(scr + Cfg::S_WIN),
                                     tbase + Cfg::T_V + (uint32_t(32 * q4) << 16));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(vdone);
            }
            if (COMMIT) pwait(&kpfull[iu & 1], (iu >> 1) & 1, abort_flag, a.status, lim);
            pwait(&ufull[us], (iu / NXS) & 1, abort_flag, a.status, lim);
            if constexpr (!TREE && TMAX >= 16)   // 16-position chains: Gram block and records here
                chain_gram_fold<Cfg>(warp - 10, lane, tid - 320, 2, T,
                                     smem + Cfg::OFF_X + size_t(us) * Cfg::X_BYTES,
                                     const_cast<float*>(meta), scr + Cfg::S_GRAM, scr + Cfg::S_GP);
            if constexpr (GDK)                   // per-key-channel gates: the decayed Gram here
                gdk_gram_records<Cfg>(tid - 320, kh, Hv, T, 2, a.g + lb * T * size_t(Hv) * D,
                                      const_cast<float*>(meta));
            if (COMMIT && n > 0) {
                const int et = tid - 320, ew = warp - 10;
                // the new conv-state rows, stashed by the prep warps, to HBM as 16-byte vectors
                const IO* cw_s = reinterpret_cast<const IO*>(meta + Cfg::M_CW);
                IO* cso = static_cast<IO*>(a.conv_state_out) + lb * size_t(W - 1) * C;
                constexpr int EPV = 16 / Cfg::ES, VPR = D / EPV;      // elements per vector, vectors per row
                const int nvec = Cfg::NPARTS * (W - 1) * VPR;
                for (int v = et; v < nvec; v += 128) {
                    const int part = v / ((W - 1) * VPR), rem = v - part * (W - 1) * VPR;
                    const int r = rem / VPR, c16 = rem - r * VPR;
                    const int cb = part == 0 ? kh * D
                                 : part == 1 ? Hk * D + kh * D : 2 * Hk * D + (kh * G + part - 2) * D;
                    *reinterpret_cast<uint4*>(cso + size_t(r) * C + cb + c16 * EPV) =
                        *reinterpret_cast<const uint4*>(cw_s + (size_t(part) * 3 + r) * D + c16 * EPV);
                }
                // GP[s][c] = k'_s · X_c on the warp tensor path (3xTF32), as the prep's Gram block:
                // warp ew takes channels 32 ew .. 32 ew + 31, partials reduced over the 4 warps
                const int gq = lane >> 2, gt4 = lane & 3;
                const unsigned char* Xb = smem + Cfg::OFF_X + size_t(us) * Cfg::X_BYTES;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int ks = 0; ks < 4; ++ks) {
                    const int ch = 32 * ew + 8 * ks + gt4;
                    float av[4];
                    av[0] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch, XKB));
                    av[2] = *reinterpret_cast<const float*>(Xb + sw128_off(gq, ch + 4, XKB));
                    av[1] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch, XKB)) : 0.f;
                    av[3] = (gq + 8 < 2 * TMAX) ? *reinterpret_cast<const float*>(Xb + sw128_off(gq + 8, ch + 4, XKB)) : 0.f;
                    uint32_t ahi[4], alo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float h = tf32_trunc(av[e]);
                        ahi[e] = __float_as_uint(h);
                        alo[e] = __float_as_uint(tf32_trunc(av[e] - h));
                    }
                    const float kv0 = gq < n ? kp[Cfg::KP_K + gq * Cfg::KP_KS + ch] : 0.f;
                    const float kv1 = gq < n ? kp[Cfg::KP_K + gq * Cfg::KP_KS + ch + 4] : 0.f;
                    const float kh0 = tf32_trunc(kv0), kh1 = tf32_trunc(kv1);
                    const uint32_t kl0 = __float_as_uint(tf32_trunc(kv0 - kh0));
                    const uint32_t kl1 = __float_as_uint(tf32_trunc(kv1 - kh1));
                    mma_tf32_16x8x8(acc, ahi, __float_as_uint(kh0), __float_as_uint(kh1));
                    mma_tf32_16x8x8(acc, ahi, kl0, kl1);
                    mma_tf32_16x8x8(acc, alo, __float_as_uint(kh0), __float_as_uint(kh1));
                }
                float* egp = scr + Cfg::S_EGP;
                float* e4 = egp + ew * 128;
                e4[gq * 8 + 2 * gt4] = acc[0];
                e4[gq * 8 + 2 * gt4 + 1] = acc[1];
                e4[(gq + 8) * 8 + 2 * gt4] = acc[2];
                e4[(gq + 8) * 8 + 2 * gt4 + 1] = acc[3];
                named_bar(2, 128);
                {
                    const int m = et >> 3, nn = et & 7;
                    if (m < 2 * TMAX && nn < TMAX)
                        const_cast<float*>(meta)[Cfg::M_GP + nn * 2 * TMAX + m] =
                            egp[et] + egp[128 + et] + egp[256 + et] + egp[384 + et];
                }
                named_bar(2, 128);
            }
            const int ps = iu % Cfg::NUS;
            if constexpr (Cfg::BIG) {
                // δ and o of both value heads, each as one triangular solve on the tensor core: the
                // recurrence δ_t = β_t (v_t − γ_t (c0k_t P_k[t] + Σ_x CK[t][x] δ_x)) over the
                // 128 value rows at once is δ = M r with M = (I + diag(βγ) CK)⁻¹ and
                // r_t = β_t (v_t − γ_t c0k_t P_k[t]); the outputs are o = e ∘ P_q + N r with
                // N = scale (diag(k·q) + diag(γ) CQ) M and e_t = scale γ_t c0q_t. CK and CQ are zero
                // off each node's ancestors, so M and N are too: row t of M (and of N) lives on t's
                // root path. Thread (head jc, node tn, part) solves it by back-substitution up that
                // path p_0 = tn, p_1 = parent, ..: v_0 = 1 and v_j = −Σ_{k<j} v_k L[p_k][p_j] for M,
                // v_0 = scale k·q_tn and v_j = scale γ_tn CQ[tn][p_j] − Σ_{k<j} v_k L[p_k][p_j] for N,
                // with L[p_k][p_j] = β γ of p_k times CK[p_k][p_j] (y (I + L) = e_tn, z (I + L) = q_tn).
                // Threads past the unit's heads idle. This runs while the unit's products are on the
                // tensor core.
                const int e_t = tid - 320, jc = e_t >> 6, tn = (e_t >> 1) & 31, part = e_t & 1;
                float* mw = const_cast<float*>(meta);
                if (jc >= G) {
                    named_bar(2, 128);
                } else {
                    const float* ck = meta + Cfg::M_REC + jc * Cfg::RJ;
                    const float* fb = meta + Cfg::M_FLD + jc * Cfg::FJ;
                    const int* pm = reinterpret_cast<const int*>(meta + Cfg::M_PAR);
                    // paths of up to PR nodes in registers; a longer one (a deeper tree) walks
                    // thread-local arrays
                    constexpr int PR = 8;
                    int pr[PR];
                    float vr[PR];
                    int dr = 0;
                    bool deep = false;
                    int pn[TMAX];
                    float vv[TMAX], uu[TMAX];
                    int d = 0;
                    if (tn < T) {
                        const float gt = fb[Cfg::F_GAM + tn];
                        const float v0 = part ? scale * fb[Cfg::F_KQ + tn] : 1.f;
                        int y = pm[tn];
                        pr[0] = tn;
#pragma unroll
                        for (int j = 1; j < PR; ++j) {
                            pr[j] = y >= 0 ? y : 0;
                            dr += y >= 0 ? 1 : 0;
                            y = y >= 0 ? pm[y] : -1;
                        }
                        dr += 1;
                        deep = y >= 0;
                        if (!deep) {
                            float ur[PR];
                            vr[0] = v0;
                            ur[0] = v0 * (fb[Cfg::F_BET + tn] * gt);
#pragma unroll
                            for (int j = 1; j < PR; ++j) {
                                const int yj = pr[j];
                                const float* crow = ck + Cfg::F_CKT + yj * TMAX;
                                float acc = part ? scale * (gt * ck[Cfg::F_CQT + yj * TMAX + tn]) : 0.f;
#pragma unroll
                                for (int k = 0; k < j; ++k) acc = fmaf(-ur[k], crow[pr[k]], acc);
                                vr[j] = acc;
                                ur[j] = j < dr ? acc * (fb[Cfg::F_BET + yj] * fb[Cfg::F_GAM + yj]) : 0.f;
                            }
                        } else {
                            pn[0] = tn;
                            vv[0] = v0;
                            uu[0] = v0 * (fb[Cfg::F_BET + tn] * gt);
                            d = 1;
                            for (int y2 = pm[tn]; y2 >= 0 && d < TMAX; y2 = pm[y2], ++d) {
                                const float* crow = ck + Cfg::F_CKT + y2 * TMAX;
                                float acc = part ? scale * (gt * ck[Cfg::F_CQT + y2 * TMAX + tn]) : 0.f;
                                for (int k = 0; k < d; ++k) acc = fmaf(-uu[k], crow[pn[k]], acc);
                                pn[d] = y2;
                                vv[d] = acc;
                                uu[d] = acc * (fb[Cfg::F_BET + y2] * fb[Cfg::F_GAM + y2]);
                            }
                        }
                    }
                    named_bar(2, 128);     // every CK / CQ entry has been read: head 1's tile goes there
                    unsigned char* tile = reinterpret_cast<unsigned char*>(mw + (jc == 0 ? Cfg::M_UT : Cfg::M_REC));
                    const int row = (part ? 32 : 0) + tn;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        *reinterpret_cast<float4*>(tile + sw128_off(row, 4 * c, 0)) = make_float4(0.f, 0.f, 0.f, 0.f);
                        *reinterpret_cast<float4*>(tile + sw128_off(64 + row, 4 * c, 0)) = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    if (!deep) {
#pragma unroll
                        for (int k = 0; k < PR; ++k) {
                            if (k < dr) {
                                const float v = vr[k];
                                *reinterpret_cast<float*>(tile + sw128_off(row, pr[k], 0)) = v;
                                *reinterpret_cast<float*>(tile + sw128_off(64 + row, pr[k], 0)) = v - tf32_trunc(v);
                            }
                        }
                    } else {
                        for (int k = 0; k < d; ++k) {
                            const float v = vv[k];
                            *reinterpret_cast<float*>(tile + sw128_off(row, pn[k], 0)) = v;
                            *reinterpret_cast<float*>(tile + sw128_off(64 + row, pn[k], 0)) = v - tf32_trunc(v);
                        }
                    }
                    fence_async_smem();
                }
                pwait(&tfull[ps], (iu / Cfg::NUS) & 1, abort_flag, a.status, lim);
                tc_fence_after();
                const uint32_t lq = uint32_t(32 * q4) << 16;
                const uint32_t dt = tbase + ps * Cfg::P_COLS + lq;
                constexpr uint32_t IDESC = umma_idesc_tf32(128, 64);
                const size_t ostep = size_t(Hv) * D;                 // next position, same head
#pragma unroll 1
                for (int j = 0; j < G; ++j) {
                    const int h = kh * G + j;
                    const float* fb = meta + Cfg::M_FLD + j * Cfg::FJ;
                    {
                        // A operand: r (zero past T) as hi (raw fp32, read as tf32) and lo columns
                        float pk[32], vv[32];
                        tmem_ld32(dt + j * S * Cfg::CH_COLS, pk);
#pragma unroll
                        for (int sc = 1; sc < S; ++sc) {           // the odd K-steps' chain
                            float pp[32];
                            tmem_ld32(dt + (j * S + sc) * Cfg::CH_COLS, pp);
#pragma unroll
                            for (int e = 0; e < 32; ++e) pk[e] += pp[e];
                        }
                        tmem_ld32(tbase + Cfg::T_V + lq + j * TMAX, vv);
                        uint32_t rh[32], rl[32];
#pragma unroll
                        for (int t4 = 0; t4 < TMAX / 4; ++t4) {
                            const float4 b4 = *reinterpret_cast<const float4*>(fb + Cfg::F_BET + 4 * t4);
                            const float4 g4 = *reinterpret_cast<const float4*>(fb + Cfg::F_GAM + 4 * t4);
                            const float4 c4 = *reinterpret_cast<const float4*>(fb + Cfg::F_C0K + 4 * t4);
                            const float bs[4] = {b4.x, b4.y, b4.z, b4.w}, gs[4] = {g4.x, g4.y, g4.z, g4.w},
                                        cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = 4 * t4 + e;
                                const float r = bs[e] * (vv[t] - gs[e] * (cs[e] * pk[t]));
                                const float rr = t < T ? r : 0.f;
                                rh[t] = __float_as_uint(rr);
                                rl[t] = __float_as_uint(rr - tf32_trunc(rr));
                            }
                        }
                        tmem_st32(tbase + Cfg::T_R + lq, rh);
                        tmem_st32(tbase + Cfg::T_R + lq + 32, rl);
                    }
                    {
                        // accumulator: [0 | e ∘ P_q]
                        float pq[32];
                        tmem_ld32(dt + j * S * Cfg::CH_COLS + TMAX, pq);
#pragma unroll
                        for (int sc = 1; sc < S; ++sc) {
                            float pp[32];
                            tmem_ld32(dt + (j * S + sc) * Cfg::CH_COLS + TMAX, pp);
#pragma unroll
                            for (int e = 0; e < 32; ++e) pq[e] += pp[e];
                        }
                        if (j == G - 1) {          // the unit's P slot has been read
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[ps]);
                        }
                        uint32_t zq[32], eq[32];
#pragma unroll
                        for (int t4 = 0; t4 < TMAX / 4; ++t4) {
                            const float4 g4 = *reinterpret_cast<const float4*>(fb + Cfg::F_GAM + 4 * t4);
                            const float4 c4 = *reinterpret_cast<const float4*>(fb + Cfg::F_C0Q + 4 * t4);
                            const float gs[4] = {g4.x, g4.y, g4.z, g4.w}, cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int t = 4 * t4 + e;
                                const float ev = scale * (gs[e] * cs[e]) * pq[t];
                                zq[t] = 0u;
                                eq[t] = __float_as_uint(t < T ? ev : 0.f);
                            }
                        }
                        tmem_st32(tbase + Cfg::T_D + lq, zq);
                        tmem_st32(tbase + Cfg::T_D + lq + 32, eq);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar(2, 128);     // r, the accumulator and this head's B tile are in place
                    if (warp == 10) {
                        tc_fence_after();
                        const uint64_t bd = umma_desc_sw128(smem_u32(mw + (j == 0 ? Cfg::M_UT : Cfg::M_REC)));
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t bk = bd + uint64_t((ks * 32) >> 4);
                            const uint64_t bl = bk + uint64_t((64 * 128) >> 4);
                            umma_tf32_ts_warp(tbase + Cfg::T_D, tbase + Cfg::T_R + ks * 8, bk, IDESC, 1u);
                            umma_tf32_ts_warp(tbase + Cfg::T_D, tbase + Cfg::T_R + ks * 8, bl, IDESC, 1u);
                            umma_tf32_ts_warp(tbase + Cfg::T_D, tbase + Cfg::T_R + 32 + ks * 8, bk, IDESC, 1u);
                        }
                        umma_commit_warp(ebar);
                    }
                    pwait(ebar, uint32_t(iu * G + j) & 1u, abort_flag, a.status, lim);   // G commits a unit
                    tc_fence_after();
                    float* tdp = a.tape_delta + (lb * T * Hv + h) * size_t(D) + i;
                    IO* op = out + (lb * T * Hv + h) * size_t(D) + i;
                    {
                        float dv[32];
                        tmem_ld32(tbase + Cfg::T_D + lq, dv);
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            st_global_if(tdp, dv[t], t < T);
                            tdp = opaque_advance(tdp, ostep);
                        }
                    }
                    {
                        float ov[32];
                        tmem_ld32(tbase + Cfg::T_D + lq + 32, ov);
#pragma unroll
                        for (int t = 0; t < TMAX; ++t) {
                            st_global_if(op, ov[t], t < T);
                            op = opaque_advance(op, ostep);
                        }
                    }
                }
            } else {
            pwait(&tfull[ps], (iu / Cfg::NUS) & 1, abort_flag, a.status, lim);
            tc_fence_after();
            const uint32_t dt = tbase + ps * Cfg::P_COLS + (uint32_t(32 * q4) << 16);
#pragma unroll 1
            for (int j = 0; j < G; ++j) {
                const int h = kh * G + j;
                {
                // P row i of this head: S_hi·X_hi + S_hi·X_lo + S_lo·X_hi over its chains
                float pr[NP];
#pragma unroll
                for (int c = 0; c < NP; ++c) pr[c] = 0.f;
#pragma unroll
                for (int sc = 0; sc < S; ++sc) {
                    const uint32_t ca = dt + (j * S + sc) * Cfg::CH_COLS;
#pragma unroll
                    for (int off = 0; off < 3 * NP; off += 16) {     // X_hi, X_lo, lo-pass blocks
                        float part[16];
                        tmem_ld16(ca + off, part);
                        const int c0 = off % NP;
#pragma unroll
                        for (int c = 0; c < 16; ++c) pr[c0 + c] += part[c];
                    }
                }
                if (j == G - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[ps]);
                }
                if (COMMIT && n > 0) {
                    // the committed state's products: Γ (S_0 X) + Σ_s (c_s δ_s[i]) (k'_s · X)
                    const float gm = kp[Cfg::KP_GAM + j];
#pragma unroll
                    for (int c = 0; c < 2 * TMAX; ++c) pr[c] *= gm;
#pragma unroll 1
                    for (int s2 = 0; s2 < n; ++s2) {
                        const float av = kp[Cfg::KP_C + j * TMAX + s2] * kp[Cfg::KP_DL + (j * TMAX + s2) * Cfg::KP_KS + i];
                        const float4* gpr = reinterpret_cast<const float4*>(meta + Cfg::M_GP + s2 * 2 * TMAX);
#pragma unroll
                        for (int c4 = 0; c4 < 2 * TMAX / 4; ++c4) {
                            const float4 gv = gpr[c4];
                            pr[4 * c4] = fmaf(av, gv.x, pr[4 * c4]);
                            pr[4 * c4 + 1] = fmaf(av, gv.y, pr[4 * c4 + 1]);
                            pr[4 * c4 + 2] = fmaf(av, gv.z, pr[4 * c4 + 2]);
                            pr[4 * c4 + 3] = fmaf(av, gv.w, pr[4 * c4 + 3]);
                        }
                    }
                }
                const float* R = meta + Cfg::M_REC + j * TMAX * RS;
                const float* vv = meta + Cfg::M_V + size_t(j) * TMAX * D + i;
                // every position is computed (no branch in the unrolled body); positions t >= T
                // are never stored and feed only later positions >= T
                const size_t ostep = size_t(Hv) * D;
                float* tdp = a.tape_delta + (lb * T * Hv + h) * size_t(D) + i;
                IO* op = out + (lb * T * Hv + h) * size_t(D) + i;
                float dl[TMAX];
#pragma unroll
                for (int t = 0; t < TMAX; ++t) {
                    {
                        const float4 hd = *reinterpret_cast<const float4*>(R + t * RS);  // c0 γ β kq
                        float sk, sq;
                        if constexpr (TREE) {
                            const float4 h2 = *reinterpret_cast<const float4*>(R + t * RS + 4);  // c0q mask
                            const unsigned gmask = __float_as_uint(h2.y);
                            sk = hd.x * pr[t];
                            sq = h2.x * pr[TMAX + t];
#pragma unroll
                            for (int q = 0; q < (t + 3) / 4; ++q) {
                                if (!((gmask >> q) & 1u)) continue;       // no ancestor in 4q .. 4q+3
                                const float4 x = *reinterpret_cast<const float4*>(R + t * RS + Cfg::HDR + 4 * q);
                                const float4 y = *reinterpret_cast<const float4*>(R + t * RS + Cfg::HDR + TMAX + 4 * q);
                                const float xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    if (4 * q + e < t) {
                                        sk = fmaf(xs[e], dl[4 * q + e], sk);
                                        sq = fmaf(ys[e], dl[4 * q + e], sq);
                                    }
                                }
                            }
                        } else {
                            float ck[TMAX], cq[TMAX];
#pragma unroll
                            for (int q = 0; q < (t + 3) / 4; ++q) {
                                const float4 x = *reinterpret_cast<const float4*>(R + t * RS + 4 + 4 * q);
                                const float4 y = *reinterpret_cast<const float4*>(R + t * RS + 4 + TMAX + 4 * q);
                                ck[4 * q] = x.x; ck[4 * q + 1] = x.y; ck[4 * q + 2] = x.z; ck[4 * q + 3] = x.w;
                                cq[4 * q] = y.x; cq[4 * q + 1] = y.y; cq[4 * q + 2] = y.z; cq[4 * q + 3] = y.w;
                            }
                            sk = hd.x * pr[t];
                            sq = hd.x * pr[TMAX + t];
#pragma unroll
                            for (int s = 0; s < t; ++s) {
                                sk = fmaf(ck[s], dl[s], sk);
                                sq = fmaf(cq[s], dl[s], sq);
                            }
                        }
                        const float u = hd.y * sk;
                        const float d = hd.z * (vv[t * D] - u);
                        dl[t] = d;
                        const float o = scale * fmaf(d, hd.w, hd.y * sq);
                        st_global_if(tdp, d, t < T);
                        st_global_if(op, o, t < T);
                        tdp = opaque_advance(tdp, ostep);
                        op = opaque_advance(op, ostep);
                    }
                }
                }
            }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&uempty[us]);
                if (COMMIT) mbar_arrive(&kpempty[iu & 1]);
            }
        }
        if constexpr (Cfg::BIG) {
            // every product this warp issued has completed before TMEM is released
            if (warp == 10) {
                umma_commit_warp(edone);
                volatile int no_abort = 0;
                pwait_warp(edone, 0, &no_abort, a.status);
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

template <typename IO, int TMAX, int G, bool COMMIT, bool TREE = false, bool GDK = false>
cudaError_t launch_verify_pipe_t(const VerifyArgs& a, const VerifyMaps& m, cudaStream_t stream) {
    using Cfg = PipeCfg<IO, TMAX, G, COMMIT, TREE, GDK>;
    auto kern = gdn_verify_pipe_kernel<IO, TMAX, G, COMMIT, TREE, GDK>;
    cudaError_t e = smem_optin(reinterpret_cast<const void*>(kern), Cfg::SMEM);
    if (e != cudaSuccess) return e;
    int nsm = 0;
    e = device_sm_count(&nsm);
    if (e != cudaSuccess) return e;
    const int n_units = a.L * a.B * a.Hk;
    const int grid = n_units < nsm ? n_units : nsm;
    kern<<<grid, Cfg::NTHR, Cfg::SMEM, stream>>>(a, m.state, m.qkv, m.conv_state,
                                                  COMMIT ? m.qkv_prev : m.qkv, n_units);
    return cudaGetLastError();
}

// The pipelined kernel serves the Qwen3.6 head shape (chains up to 16 positions, trees up to 32
// nodes) with one gate per value head, and chains up to 8 positions with one gate per key channel;
// everything else uses the per-head kernel.
template <typename IO>
bool verify_pipe_eligible(const VerifyArgs& a, const VerifyMaps& m, int D, bool tree, bool commit) {
    const int tmax = commit ? 8 : (tree ? 32 : 16);
    return m.inputs_ok && (!a.gate_dk || (!tree && !commit && a.T <= 8)) && !(tree && commit) &&
           D == 128 && sizeof(IO) == 2 && a.T <= tmax && (a.Hv == a.Hk || a.Hv == 2 * a.Hk);
}

template <typename IO, int TMAX, bool COMMIT, bool TREE, bool GDK = false>
cudaError_t launch_verify_pipe_g(const VerifyArgs& a, const VerifyMaps& m, cudaStream_t s) {
    return a.Hv == a.Hk ? launch_verify_pipe_t<IO, TMAX, 1, COMMIT, TREE, GDK>(a, m, s)
                        : launch_verify_pipe_t<IO, TMAX, 2, COMMIT, TREE, GDK>(a, m, s);
}

template <typename IO, bool COMMIT>
cudaError_t launch_verify_pipe(const VerifyArgs& a, const VerifyMaps& m, bool tree, cudaStream_t s) {
    if constexpr (!COMMIT) {
        if (a.gate_dk)   // chains of T <= 8 (verify_pipe_eligible)
            return a.T <= 4 ? launch_verify_pipe_g<IO, 4, false, false, true>(a, m, s)
                            : launch_verify_pipe_g<IO, 8, false, false, true>(a, m, s);
        if (tree) {
            if (a.T <= 8) return launch_verify_pipe_g<IO, 8, false, true>(a, m, s);
            if (a.T <= 16) return launch_verify_pipe_g<IO, 16, false, true>(a, m, s);
            return launch_verify_pipe_g<IO, 32, false, true>(a, m, s);
        }
    }
    if (a.T <= 4) return launch_verify_pipe_g<IO, 4, COMMIT, false>(a, m, s);
    if (COMMIT || a.T <= 8) return launch_verify_pipe_g<IO, 8, COMMIT, false>(a, m, s);
    if constexpr (!COMMIT) return launch_verify_pipe_g<IO, 16, false, false>(a, m, s);
    return cudaErrorNotSupported;
}

}  // namespace gdn
