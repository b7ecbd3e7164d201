// accept.cu — spec_accept / spec_accept_tree kernels (sm_103a).
//
// Greedy ("Phase 25: 三种投机解码方法对比", §2 algorithm; colibrì analysis ch.08 §5 greedy path):
//   accept the longest prefix of drafts equal to the row argmax, then emit the argmax of the first
//   unmatched row (the correction) or of the bonus row.
// Sampling (colibrì analysis ch.08 §5, Leviathan rejection sampling with point-mass drafts):
//   accept draft i with probability p_i(draft_i); on the first rejection ban the draft, renormalise
//   and resample; if every draft is accepted sample the bonus row. p is realised by integer
//   weights w = floor(2^32 · 2^((l − max)·c)) so the decisions are exact and order-independent.
//
// Structure (HBM-bound: every logits row is read once, sampling re-reads it from L2):
//   K1 rowmax   grid (rows, chunks): chunk argmax, lowest index on ties, as a packed u64 key.
//               A NaN logit is never taken (it counts as −∞); a row of NaN / −∞ gives index 0.
//   K2 weights  grid (rows, chunks): chunk weight sums (u64) and the draft token's weight.
//   K3 scan     one CTA per sequence: the sequential accept decisions of the pages' loop; a
//               rejection or the bonus searches one chunk for the sampled token.
// Every vocabulary row is split into CH chunks of CS elements; rows start on 16-byte boundaries
// and are read with 16-byte vector loads.
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"

namespace gdn {

constexpr int kAccThreads = 256;

// ---------------------------------------------------------------- logits element access
template <typename LT> struct LogitVec;
template <> struct LogitVec<__nv_bfloat16> {
    static constexpr int N = 8;   // elements per 16-byte vector
    __device__ static __forceinline__ void load(const __nv_bfloat16* p, float (&v)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ float one(const __nv_bfloat16* p) {
        return __bfloat162float(p[0]);
    }
};
template <> struct LogitVec<float> {
    static constexpr int N = 4;
    __device__ static __forceinline__ void load(const float* p, float (&v)[4]) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
    __device__ static __forceinline__ float one(const float* p) { return __ldg(p); }
};

// order-preserving map of float bits to u32, and the packed (value, lowest index) key
__device__ __forceinline__ uint32_t ord_f32(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long pack_key(float v, int idx) {
    return (static_cast<unsigned long long>(ord_f32(v)) << 32) | (0xffffffffu - uint32_t(idx));
}
__device__ __forceinline__ int key_index(unsigned long long k) {
    return int(0xffffffffu - uint32_t(k & 0xffffffffull));
}

// ---------------------------------------------------------------- integer-weight contract
// The integer weight w = floor(2^32 · 2^x), x = (l − m)·c ≤ 0, with this library's 2^x: Cody–Waite
// reduction x = n + f (n = rint(x), f in [-1/2, 1/2]), the degree-7 Taylor polynomial p of 2^f
// (coefficients (ln 2)^k / k! rounded to fp32, Horner with fused multiply-adds), 2^x = p · 2^n,
// zero for n < -64. p lies in [2^-1/2, 1] (a normal fp32 with 24-bit significand M and biased
// exponent E), and p · 2^n · 2^32 is exact in fp32, so w = floor(M · 2^sh), sh = E − 127 + n + 9,
// a shift with no float-to-integer conversion: with a = M · 2^8 (32 bits), w = a >> (8 − sh) for
// sh ≤ 8 (a right shift by 32 or more gives 0, which covers n < -64), and w = 2a for sh = 9 (p = 1,
// n = 0: the row maximum). n comes from the bits of x + 1.5·2^23 (round to nearest even, exact
// for |x| < 2^22; x is clamped to [-100, 0] first, where every weight is 0 below -64.5).
// A NaN logit counts as −∞ (weight 0: fmaxf turns a NaN x into -100), and so does a NaN x from a
// −∞ or NaN logit against a −∞ maximum. The row max never is NaN (the max passes skip NaN).
__device__ __forceinline__ unsigned long long weight_of(float l, float m, float c) {
    const float x = fmaxf(__fmul_rn(__fsub_rn(l, m), c), -100.0f);
    const float t = __fadd_rn(x, 12582912.0f);
    const int n = __float_as_int(t) - 0x4B400000;       // rint(x)
    const float f = __fsub_rn(x, __fsub_rn(t, 12582912.0f));
    float p = 0x1.ffcbfcp-17f;
    p = __fmaf_rn(p, f, 0x1.430912p-13f);
    p = __fmaf_rn(p, f, 0x1.5d87fep-10f);
    p = __fmaf_rn(p, f, 0x1.3b2ab6p-7f);
    p = __fmaf_rn(p, f, 0x1.c6b08ep-5f);
    p = __fmaf_rn(p, f, 0x1.ebfbe0p-3f);
    p = __fmaf_rn(p, f, 0x1.62e430p-1f);
    p = __fmaf_rn(p, f, 1.0f);
    const uint32_t pb = __float_as_uint(p);
    const uint32_t a = (pb << 8) | 0x80000000u;          // M · 2^8
    const int s = 126 - int(pb >> 23) - n;              // 8 − sh, >= -1
    uint32_t w;
    asm("shr.b32 %0, %1, %2;" : "=r"(w) : "r"(a), "r"(s));   // amounts >= 32 give 0
    return s < 0 ? (static_cast<unsigned long long>(a) << 1) : static_cast<unsigned long long>(w);
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11), counter (c0..c3), key (k0, k1).
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    }
}

// r = floor(U · Z / 2^128) with U the 128-bit Philox output for counter (round, seq, row, purpose).
__device__ __forceinline__ unsigned long long draw_uniform(uint64_t seed, uint32_t round,
                                                           uint32_t seq, uint32_t row,
                                                           uint32_t purpose,
                                                           unsigned long long Z) {
    uint32_t c[4] = {round, seq, row, purpose};
    philox4x32_10(c, uint32_t(seed), uint32_t(seed >> 32));
    const unsigned long long Uh = (static_cast<unsigned long long>(c[3]) << 32) | c[2];
    const unsigned long long Ul = (static_cast<unsigned long long>(c[1]) << 32) | c[0];
    const unsigned long long lo = Uh * Z, hi = __umul64hi(Uh, Z);
    const unsigned long long add = __umul64hi(Ul, Z);
    const unsigned long long lo2 = lo + add;
    return hi + (lo2 < lo ? 1ull : 0ull);
}

// ---------------------------------------------------------------- block reductions
__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v,
                                                            unsigned long long* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, v, o);
        v = x > v ? x : v;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (kAccThreads / 32) ? sh[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xffffffffu, v, o);
            v = x > v ? x : v;
        }
    }
    return v;   // valid in thread 0
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < (kAccThreads / 32) ? sh[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    }
    return v;   // valid in thread 0
}

// exclusive prefix sum over the block; returns this thread's prefix, *total = block sum
__device__ __forceinline__ unsigned long long block_exscan_u64(unsigned long long v,
                                                               unsigned long long* sh,
                                                               unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) sh[warp] = inc;
    __syncthreads();
    unsigned long long base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kAccThreads / 32; ++w) {
        const unsigned long long s = sh[w];
        if (w < warp) base += s;
        tot += s;
    }
    __syncthreads();
    *total = tot;
    return base + inc - v;
}

__device__ __forceinline__ const void* row_ptr(const AcceptArgs& a, int b, int i, int esize) {
    return static_cast<const char*>(a.logits) +
           (size_t(b) * a.seq_stride + size_t(i) * a.row_stride) * esize;
}

// ---------------------------------------------------------------- K1: chunk argmax
template <typename LT>
__global__ void __launch_bounds__(kAccThreads) accept_rowmax_kernel(const AcceptArgs a) {
    using LV = LogitVec<LT>;
    __shared__ unsigned long long sh[kAccThreads / 32];
    const int RS = a.N + 1;
    const int r = blockIdx.x, ch = blockIdx.y;
    const int b = r / RS, i = r - b * RS;
    const LT* row = static_cast<const LT*>(row_ptr(a, b, i, sizeof(LT)));
    const int lo = ch * a.CS, hi = min(a.V, lo + a.CS);
    // (−inf, lo) is a valid start: if the whole chunk is −inf, element lo is its argmax
    float bv = -INFINITY;
    int bi = lo;
    const int vec_hi = lo + (hi - lo) / LV::N * LV::N;
#pragma unroll 4
    for (int v0 = lo + threadIdx.x * LV::N; v0 < vec_hi; v0 += kAccThreads * LV::N) {
        float x[LV::N];
        LV::load(row + v0, x);
#pragma unroll
        for (int k = 0; k < LV::N; ++k)
            if (x[k] > bv) { bv = x[k]; bi = v0 + k; }
    }
    for (int v = vec_hi + threadIdx.x; v < hi; v += kAccThreads) {
        const float x = LV::one(row + v);
        if (x > bv || (x == bv && v < bi)) { bv = x; bi = v; }
    }
    unsigned long long key = pack_key(bv, bi);
    key = block_max_u64(key, sh);
    if (threadIdx.x == 0) a.ws_key[size_t(r) * a.CH + ch] = key;
}

__device__ __forceinline__ unsigned long long row_best_key(const AcceptArgs& a, int r) {
    unsigned long long best = 0;
    for (int c = 0; c < a.CH; ++c) {
        const unsigned long long k = a.ws_key[size_t(r) * a.CH + c];
        best = k > best ? k : best;
    }
    return best;
}

// ---------------------------------------------------------------- K2: chunk weight sums
// One warp per tile of 32 consecutive 16-byte vectors (coalesced): the tile's exact u64 weight
// sum goes to ws_tile (so a later search needs only one tile), the chunk sum to ws_sum, the draft
// token's weight to ws_wd.
template <typename LT>
__global__ void __launch_bounds__(kAccThreads) accept_weights_kernel(const AcceptArgs a) {
    using LV = LogitVec<LT>;
    constexpr int TILE = 32 * LV::N;
    __shared__ unsigned long long sh[kAccThreads / 32];
    __shared__ float s_m;
    const int RS = a.N + 1;
    const int r = blockIdx.x, ch = blockIdx.y;
    const int b = r / RS, i = r - b * RS;
    if (threadIdx.x == 0) s_m = unord_f32(uint32_t(row_best_key(a, r) >> 32));
    __syncthreads();
    const float m = s_m, c = a.c;
    const int d = (i < a.N) ? a.drafts[size_t(b) * a.N + i] : -1;
    const LT* row = static_cast<const LT*>(row_ptr(a, b, i, sizeof(LT)));
    const int lo = ch * a.CS, hi = min(a.V, lo + a.CS);
    const int nt = (hi - lo + TILE - 1) / TILE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned long long* tiles = a.ws_tile + (size_t(r) * a.CH + ch) * a.NT;
    unsigned long long sum = 0;
    for (int t = warp; t < nt; t += kAccThreads / 32) {
        const int v0 = lo + t * TILE + lane * LV::N;
        unsigned long long ts = 0;
        if (v0 + LV::N <= hi) {
            float x[LV::N];
            LV::load(row + v0, x);
#pragma unroll
            for (int k = 0; k < LV::N; ++k) {
                const unsigned long long w = weight_of(x[k], m, c);
                ts += w;
                if (v0 + k == d) a.ws_wd[r] = w;
            }
        } else {
            for (int k = 0; k < LV::N && v0 + k < hi; ++k) {
                const unsigned long long w = weight_of(LV::one(row + v0 + k), m, c);
                ts += w;
                if (v0 + k == d) a.ws_wd[r] = w;
            }
        }
        sum += ts;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
        if (lane == 0) tiles[t] = ts;
    }
    sum = block_sum_u64(sum, sh);
    if (threadIdx.x == 0) a.ws_sum[size_t(r) * a.CH + ch] = sum;
}

// ---------------------------------------------------------------- K3 helpers
// smallest v in chunk `ch` of row (b, i) whose in-chunk prefix of weights exceeds rr (ban = -1
// for none): the tile from a block scan of the chunk's tile sums, then one warp scans the tile's
// weights. All threads of the block call it; the result is returned to all (-1 if rr is past the
// chunk's total).
template <typename LT>
__device__ int chunk_search(const AcceptArgs& a, int b, int i, int ch, unsigned long long rr,
                            int ban, float m, unsigned long long* sh, int* s_tok) {
    using LV = LogitVec<LT>;
    constexpr int TILE = 32 * LV::N;
    __shared__ int s_tile;
    __shared__ unsigned long long s_rem;
    const int r = b * (a.N + 1) + i;
    const LT* row = static_cast<const LT*>(row_ptr(a, b, i, sizeof(LT)));
    const int lo = ch * a.CS, hi = min(a.V, lo + a.CS);
    const int nt = (hi - lo + TILE - 1) / TILE;
    const unsigned long long* tiles = a.ws_tile + (size_t(r) * a.CH + ch) * a.NT;
    const int ban_t = (ban >= lo && ban < hi) ? (ban - lo) / TILE : -1;
    const unsigned long long wban = ban_t >= 0 ? a.ws_wd[r] : 0ull;
    // 1. the tile: thread k owns tiles [k per, (k + 1) per)
    const int per = (nt + kAccThreads - 1) / kAccThreads;
    const int t_lo = min(nt, int(threadIdx.x) * per), t_hi = min(nt, t_lo + per);
    unsigned long long s = 0;
    for (int t = t_lo; t < t_hi; ++t) s += tiles[t] - (t == ban_t ? wban : 0ull);
    if (threadIdx.x == 0) { *s_tok = -1; s_tile = -1; }
    unsigned long long total;
    const unsigned long long pre = block_exscan_u64(s, sh, &total);
    if (pre <= rr && rr < pre + s) {
        unsigned long long acc = pre;
        for (int t = t_lo; t < t_hi; ++t) {
            const unsigned long long w = tiles[t] - (t == ban_t ? wban : 0ull);
            if (rr < acc + w) { s_tile = t; s_rem = rr - acc; break; }
            acc += w;
        }
    }
    __syncthreads();
    const int tile = s_tile;
    // 2. warp 0 scans the tile: lane l owns its 16-byte vector
    if (tile >= 0 && threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const unsigned long long rem = s_rem;
        const int v0 = lo + tile * TILE + lane * LV::N;
        float x[LV::N];
        if (v0 + LV::N <= hi) {
            LV::load(row + v0, x);
        } else {
#pragma unroll
            for (int k = 0; k < LV::N; ++k) x[k] = v0 + k < hi ? LV::one(row + v0 + k) : 0.f;
        }
        unsigned long long w[LV::N], ls = 0;
#pragma unroll
        for (int k = 0; k < LV::N; ++k) {
            w[k] = (v0 + k < hi && v0 + k != ban) ? weight_of(x[k], m, a.c) : 0ull;
            ls += w[k];
        }
        unsigned long long inc = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const unsigned long long lpre = inc - ls;
        if (lpre <= rem && rem < lpre + ls) {
            unsigned long long acc = lpre;
#pragma unroll
            for (int k = 0; k < LV::N; ++k) {
                acc += w[k];
                if (acc > rem) { *s_tok = v0 + k; break; }
            }
        }
    }
    __syncthreads();
    const int tok = *s_tok;
    __syncthreads();
    return tok;
}

// ---------------------------------------------------------------- K3: greedy scan
__global__ void __launch_bounds__(kAccThreads) accept_greedy_scan_kernel(const AcceptArgs a) {
    extern __shared__ int s_am[];   // [N + 1]
    __shared__ int s_bad;
    const int b = blockIdx.x, N = a.N, RS = N + 1;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < RS; i += kAccThreads) {
        s_am[i] = key_index(row_best_key(a, b * RS + i));
        if (i < N) {
            const int d = a.drafts[size_t(b) * N + i];
            if (d < 0 || d >= a.V) atomicOr(&s_bad, 1);
        }
    }
    __syncthreads();
    int32_t* out = a.out_tokens + size_t(b) * RS;
    if (s_bad) {
        for (int i = threadIdx.x; i < RS; i += kAccThreads) out[i] = -1;
        if (threadIdx.x == 0) { a.n_acc[b] = 0; set_status(a.status, GDN_STATUS_BAD_TOKEN); }
        return;
    }
    __shared__ int s_n;
    if (threadIdx.x == 0) {
        int n = 0;
        while (n < N && a.drafts[size_t(b) * N + n] == s_am[n]) ++n;
        s_n = n;
        a.n_acc[b] = n;
    }
    __syncthreads();
    const int n = s_n;
    for (int i = threadIdx.x; i < RS; i += kAccThreads)
        out[i] = i < n ? a.drafts[size_t(b) * N + i] : (i == n ? s_am[n] : -1);
}

// ---------------------------------------------------------------- K3: sampling scan
template <typename LT>
__global__ void __launch_bounds__(kAccThreads) accept_sample_scan_kernel(const AcceptArgs a) {
    __shared__ unsigned long long sh[kAccThreads / 32];
    __shared__ int s_bad, s_act, s_chunk, s_ban, s_tok;
    __shared__ unsigned long long s_rr;
    __shared__ float s_m;
    const int b = blockIdx.x, N = a.N, RS = N + 1;
    const int32_t* dr = a.drafts + size_t(b) * N;
    int32_t* out = a.out_tokens + size_t(b) * RS;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += kAccThreads)
        if (dr[i] < 0 || dr[i] >= a.V) atomicOr(&s_bad, 1);
    for (int i = threadIdx.x; i < RS; i += kAccThreads) out[i] = -1;
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) { a.n_acc[b] = 0; set_status(a.status, GDN_STATUS_BAD_TOKEN); }
        return;
    }
    int n = N;
    for (int i = 0; i <= N; ++i) {
        // s_act: 0 accept, 1 resample after rejection, 2 bonus sample
        if (threadIdx.x == 0) {
            const int r = b * RS + i;
            unsigned long long Z = 0;
            for (int c = 0; c < a.CH; ++c) Z += a.ws_sum[size_t(r) * a.CH + c];
            int act, ban = -1;
            unsigned long long rr = 0;
            if (i < N) {
                const int d = dr[i];
                const unsigned long long wd = a.ws_wd[r];
                const unsigned long long u = draw_uniform(a.seed, a.round, b, i, 0u, Z);
                if (u < wd) {
                    act = 0;
                } else {
                    act = 1;
                    ban = d;
                    Z -= wd;
                    rr = draw_uniform(a.seed, a.round, b, i, 1u, Z);
                }
            } else {
                act = 2;
                rr = draw_uniform(a.seed, a.round, b, i, 1u, Z);
            }
            if (act == 0) {
                out[i] = dr[i];
            } else {
                if (Z == 0) set_status(a.status, GDN_STATUS_EMPTY_DIST);
                int chunk = a.CH - 1;
                unsigned long long acc = 0;
                for (int c = 0; c < a.CH; ++c) {
                    unsigned long long sc = a.ws_sum[size_t(r) * a.CH + c];
                    if (ban >= c * a.CS && ban < (c + 1) * a.CS) sc -= a.ws_wd[r];
                    if (rr < acc + sc) { chunk = c; break; }
                    acc += sc;
                }
                s_chunk = chunk;
                s_rr = rr - acc;
                s_ban = ban;
                s_m = unord_f32(uint32_t(row_best_key(a, r) >> 32));
            }
            s_act = act;
        }
        __syncthreads();
        const int act = s_act;
        if (act != 0) {
            const int tok = chunk_search<LT>(a, b, i, s_chunk, s_rr, s_ban, s_m, sh, &s_tok);
            if (threadIdx.x == 0) out[i] = tok;
            if (act == 1) n = i;
            break;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) a.n_acc[b] = n;
}

// ---------------------------------------------------------------- K3: tree walk
__global__ void __launch_bounds__(kAccThreads) accept_tree_scan_kernel(const AcceptArgs a) {
    extern __shared__ int s_am[];   // [T + 1], then the parents [T] and the tokens [T]
    __shared__ int s_bad;
    const int b = blockIdx.x, T = a.N, RS = T + 1, P = a.P;
    int32_t* par = s_am + RS;       // staged in shared memory for the walk below
    int32_t* tok = par + T;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < RS; i += kAccThreads) {
        s_am[i] = key_index(row_best_key(a, b * RS + i));
        if (i < T) {
            const int32_t pv = a.parent[size_t(b) * T + i], tv = a.drafts[size_t(b) * T + i];
            par[i] = pv;
            tok[i] = tv;
            if (pv < -1 || pv >= i) atomicOr(&s_bad, 1);
            if (tv < 0 || tv >= a.V) atomicOr(&s_bad, 2);
        }
    }
    __syncthreads();
    int32_t* pth = a.path + size_t(b) * P;
    int32_t* out = a.out_tokens + size_t(b) * (P + 1);
    for (int i = threadIdx.x; i < P; i += kAccThreads) pth[i] = -1;
    for (int i = threadIdx.x; i <= P; i += kAccThreads) out[i] = -1;
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) {
            a.n_acc[b] = 0;
            set_status(a.status, ((s_bad & 1) ? GDN_STATUS_BAD_PARENT : 0u) |
                                     ((s_bad & 2) ? GDN_STATUS_BAD_TOKEN : 0u));
        }
        return;
    }
    if (threadIdx.x == 0) {
        int cur = -1, n = 0, am = s_am[0];
        while (n < P) {
            int next = -1;
            for (int v = 0; v < T; ++v)
                if (par[v] == cur && tok[v] == am) { next = v; break; }
            if (next < 0) break;
            pth[n] = next;
            out[n] = tok[next];
            ++n;
            cur = next;
            am = s_am[1 + cur];
        }
        out[n] = am;
        a.n_acc[b] = n;
    }
}

// ---------------------------------------------------------------- sampling: one cluster per sequence
// The accept loop looks at row i only once drafts 0..i-1 were accepted, so only the rows up to the
// first rejection (or the bonus row) need their weights. One cluster of CL CTAs per sequence walks
// the rows in that order. CTA k of the cluster keeps the vocabulary slice [k·SL, (k+1)·SL) of the
// current row in shared memory, each thread a contiguous run of K 16-byte vectors of it (K odd:
// the run stride then spreads a quarter warp's 16-byte reads over all banks).
//
// Each row's slice arrives by TMA bulk copies (one thread issues them; the wait on their mbarrier
// is bounded) into one of two stages, the next row's while the current one is weighed.
//
// One cluster barrier per row. Before barrier r every CTA publishes, into a slot of every peer's
// shared memory, its weight sum and draft weight of row r-1 and its maximum of row r (whose slice
// was prefetched while row r-1 was being weighed). After the barrier every thread of every CTA
// takes the same accept decision on row r-1 from the same slots; an accepted row r-1 frees its
// stage for the prefetch of row r+1, and row r's weights follow at once (its maximum is known). A
// rejection (or the bonus row) resamples: the CTA whose slice holds the draw finds the thread by a
// block scan of the per-thread sums, and that thread finds the token in its own run.
// Waits: hardware barriers (cluster, CTA), and the copies' mbarrier, whose wait gives up after about
// a second (GDN_STATUS_WAIT_TIMEOUT) and is repeated before the CTA exits.
//
// The cluster size is chosen on the host among 1..16 (above 8 where the GPU allows non-portable
// clusters): the fewest waves of B clusters (cudaOccupancyMaxActiveClusters; a GPC holds a whole
// cluster), each wave weighed as one CTA's share of a row plus a fixed part.
constexpr int kMaxCL = 16;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the copy of `local` (a shared-memory location of this CTA) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer_u64(uint32_t addr, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_peer_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// the VN logits of one 16-byte vector, as float
template <typename LT>
__device__ __forceinline__ void unpack16(const uint4& u, float (&x)[16 / sizeof(LT)]) {
    if constexpr (sizeof(LT) == 2) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else {
        x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
    }
}
// element k of a run in shared memory, as float
template <typename LT>
__device__ __forceinline__ float run_elem(const uint4* run, int k) {
    if constexpr (sizeof(LT) == 2)
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(run)[k]);
    else
        return reinterpret_cast<const float*>(run)[k];
}

struct LazySlots {
    float mx[2][kMaxCL];                 // by row parity: each CTA's slice maximum
    unsigned long long sum[2][kMaxCL];   // each CTA's weight sum
    unsigned long long wd[2][kMaxCL];    // the draft's weight (non-zero only from its slice's CTA)
};

template <typename LT>
__global__ void __launch_bounds__(1024, 1)
    accept_sample_lazy_kernel(const AcceptArgs a, const int SL, const int K) {
    constexpr int VN = LogitVec<LT>::N;       // logits per 16-byte vector
    extern __shared__ uint4 s_stage[];        // [2][blockDim.x * K]: two rows' slices, then the
                                              // sequence's N drafts (int32)
    __shared__ LazySlots slots;
    __shared__ unsigned long long s_rs[32], s_rw[32];
    __shared__ float s_rm[32];
    __shared__ uint64_t s_bar[2];             // per stage: its bulk copies landed
    __shared__ int s_bad, s_ok;
    const int NT = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = NT >> 5;
    const uint32_t rank = cluster_ctarank(), CL = cluster_nctarank();
    const int b = blockIdx.x / int(CL), N = a.N, V = a.V, RS = N + 1;
    const int lo = int(rank) * SL, hi = min(V, lo + SL);
    const int SLV = NT * K;                   // vectors per stage
    const int t0 = lo + tid * K * VN;         // this thread's first logit
    const int t1 = min(hi, t0 + K * VN);      // one past its last (t1 <= t0: an idle thread)
    // the bulk copies bring [lo, hv), a whole number of 16-byte vectors; the rest of the slice,
    // [hv, hi), is less than one vector (a vocabulary that is not a multiple of it) and is read
    // from global memory by its thread
    const uint32_t bulk_bytes = hi > lo ? (uint32_t(hi - lo) * uint32_t(sizeof(LT))) & ~15u : 0u;
    const int hv = lo + int(bulk_bytes / sizeof(LT));
    const int32_t* dr_g = a.drafts + size_t(b) * N;
    int32_t* dr = reinterpret_cast<int32_t*>(s_stage + size_t(2) * NT * K);   // [N] in shared memory

    auto row_of = [&](int i) { return static_cast<const LT*>(row_ptr(a, b, i, sizeof(LT))); };
    auto run_of = [&](int i) { return s_stage + size_t(i & 1) * SLV + size_t(tid) * K; };
    uint32_t pending = 0, pend_par = 0;       // thread 0, bit per stage: copies issued and not yet
                                              // seen landing, and their mbarrier phase parity
    auto issue_row = [&](int i) {
        if (tid == 0 && bulk_bytes) {
            uint64_t* bar = &s_bar[i & 1];
            mbar_arrive_expect_tx(bar, bulk_bytes);
            const char* src = reinterpret_cast<const char*>(row_of(i) + lo);
            char* dst = reinterpret_cast<char*>(s_stage + size_t(i & 1) * SLV);
            for (uint32_t off = 0; off < bulk_bytes; off += 32768u)
                bulk_g2s(dst + off, src + off, min(32768u, bulk_bytes - off), bar);
            pending |= 1u << (i & 1);
            pend_par = (pend_par & ~(1u << (i & 1))) | (((uint32_t(i) >> 1) & 1u) << (i & 1));
        }
    };
    // row i's copies have landed (stage i & 1 is used for the (i >> 1)-th time)
    auto wait_row = [&](int i) {
        if (!bulk_bytes) return;
        if (tid == 0) {
            const bool ok = mbar_wait_bounded(&s_bar[i & 1], uint32_t(i >> 1) & 1u);
            if (ok) pending &= ~(1u << (i & 1));
            else set_status(a.status, GDN_STATUS_WAIT_TIMEOUT);
            s_ok = ok;
        }
        __syncthreads();
        if (s_ok) (void)mbar_try_wait(&s_bar[i & 1], uint32_t(i >> 1) & 1u);   // completed: acquire
    };
    // the VN logits of vector k of this thread's run of row i (−∞ past the slice)
#define LAZY_LOAD_VEC(i_, run_, k_, x_)                                                        \
    do {                                                                                      \
        const int e0_ = t0 + (k_) * VN;                                                       \
        if (e0_ + VN <= hv) {                                                                 \
            unpack16<LT>((run_)[k_], x_);                                                     \
        } else {                                                                              \
            const LT* row_ = row_of(i_);                                                      \
            _Pragma("unroll") for (int j_ = 0; j_ < VN; ++j_)                                 \
                x_[j_] = e0_ + j_ < hi ? LogitVec<LT>::one(row_ + e0_ + j_) : -INFINITY;      \
        }                                                                                     \
    } while (0)
    // this thread's maximum of row i (NaN never wins: fmaxf returns the other operand)
    auto run_max = [&](int i) {
        const uint4* run = run_of(i);
        float mx = -INFINITY;
        for (int k = 0; k < K && t0 + k * VN < hi; ++k) {
            float x[VN];
            LAZY_LOAD_VEC(i, run, k, x);
#pragma unroll
            for (int j = 0; j < VN; ++j) mx = fmaxf(mx, x[j]);
        }
        return mx;
    };
    // publish this CTA's (sum, draft weight) of row i and maximum of row i + 1 into every peer
    auto publish = [&](int i, unsigned long long ts, unsigned long long wdv, float mxn) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ts += __shfl_xor_sync(0xffffffffu, ts, o);
            wdv += __shfl_xor_sync(0xffffffffu, wdv, o);
            mxn = fmaxf(mxn, __shfl_xor_sync(0xffffffffu, mxn, o));
        }
        if (lane == 0) { s_rs[warp] = ts; s_rw[warp] = wdv; s_rm[warp] = mxn; }
        __syncthreads();
        if (warp == 0) {
            ts = lane < nwarps ? s_rs[lane] : 0ull;
            wdv = lane < nwarps ? s_rw[lane] : 0ull;
            mxn = lane < nwarps ? s_rm[lane] : -INFINITY;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ts += __shfl_xor_sync(0xffffffffu, ts, o);
                wdv += __shfl_xor_sync(0xffffffffu, wdv, o);
                mxn = fmaxf(mxn, __shfl_xor_sync(0xffffffffu, mxn, o));
            }
            for (int r = lane; r < int(CL); r += 32) {
                if (i >= 0) {
                    st_peer_u64(peer_addr(&slots.sum[i & 1][rank], uint32_t(r)), ts);
                    st_peer_u64(peer_addr(&slots.wd[i & 1][rank], uint32_t(r)), wdv);
                }
                st_peer_f32(peer_addr(&slots.mx[(i + 1) & 1][rank], uint32_t(r)), mxn);
            }
        }
        cluster_sync_all();
    };

    if (tid == 0) {
        s_bad = 0;
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    issue_row(0);
    if (N >= 1) issue_row(1);
    // the drafts, while the first rows are in flight; one outside [0, V) ends the sequence (every
    // CTA sees the same drafts and leaves, after its copies have landed, before any peer access)
    for (int q = tid; q < N; q += NT) {
        const int32_t v = dr_g[q];
        dr[q] = v;
        if (v < 0 || v >= V) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (rank == 0) {
            int32_t* out = a.out_tokens + size_t(b) * RS;
            for (int q = tid; q < RS; q += NT) out[q] = -1;
            if (tid == 0) { a.n_acc[b] = 0; set_status(a.status, GDN_STATUS_BAD_TOKEN); }
        }
        if (tid == 0)
            for (int q = 0; q < 2; ++q)
                if ((pending >> q) & 1u) (void)mbar_wait_bounded(&s_bar[q], (pend_par >> q) & 1u);
        return;
    }
    cluster_sync_all();   // every CTA of the cluster runs before the first peer store
    wait_row(0);
    publish(-1, 0ull, 0ull, run_max(0));

    const float c = a.c;
    int i = 0, act = 0, ban = -1;
    unsigned long long rr = 0, ts = 0, wd = 0, Z = 0;
    float m = -INFINITY;
    for (;; ++i) {
        // row i's maximum is in the slots: the exact weights of this thread's run
        m = slots.mx[i & 1][0];
        for (int k = 1; k < int(CL); ++k) m = fmaxf(m, slots.mx[i & 1][k]);
        const uint4* run = run_of(i);
        ts = 0;
        int k = 0;
        for (; k + 1 < K && t0 + (k + 1) * VN < hi; k += 2) {   // two vectors at a time
            float x[VN], y[VN];
            LAZY_LOAD_VEC(i, run, k, x);
            LAZY_LOAD_VEC(i, run, k + 1, y);
            unsigned long long s0 = 0, s1 = 0;
#pragma unroll
            for (int j = 0; j < VN; ++j) {
                s0 += weight_of(x[j], m, c);
                s1 += weight_of(y[j], m, c);
            }
            ts += s0 + s1;
        }
        if (k < K && t0 + k * VN < hi) {
            float x[VN];
            LAZY_LOAD_VEC(i, run, k, x);
#pragma unroll
            for (int j = 0; j < VN; ++j) ts += weight_of(x[j], m, c);
        }
        const int d = i < N ? dr[i] : -1;
        unsigned long long wdv = 0;
        if (d >= t0 && d < t1)
            wdv = weight_of(d < hv ? run_elem<LT>(run, d - t0) : LogitVec<LT>::one(row_of(i) + d), m, c);
        float mxn = -INFINITY;
        if (i < N) {
            wait_row(i + 1);                         // prefetched while row i was weighed
            mxn = run_max(i + 1);
        }
        publish(i, ts, wdv, mxn);

        // the decision, taken identically by every thread of every CTA from the same slots
        Z = 0;
        wd = 0;
        for (int q = 0; q < int(CL); ++q) { Z += slots.sum[i & 1][q]; wd += slots.wd[i & 1][q]; }
        if (i < N) {
            const unsigned long long u = draw_uniform(a.seed, a.round, b, i, 0u, Z);
            if (u < wd) {                            // accepted: row i's stage takes row i + 2
                if (i + 2 <= N) issue_row(i + 2);
                continue;
            }
            act = 1;                                 // rejected: ban the draft, resample
            ban = d;
            Z -= wd;
            rr = draw_uniform(a.seed, a.round, b, i, 1u, Z);
        } else {
            act = 2;                                 // all accepted: the bonus row
            rr = draw_uniform(a.seed, a.round, b, i, 1u, Z);
        }
        break;
    }

    // the CTA whose slice holds rr: its prefix over the slices before it (ban removed)
    const int ban_cta = ban >= 0 ? ban / SL : -1;
    const unsigned long long wban = ban >= 0 ? wd : 0ull;
    unsigned long long pre = 0;
    for (int q = 0; q < int(rank); ++q) pre += slots.sum[i & 1][q] - (q == ban_cta ? wban : 0ull);
    const unsigned long long mine = slots.sum[i & 1][rank] - (int(rank) == ban_cta ? wban : 0ull);
    int32_t* out = a.out_tokens + size_t(b) * RS;
    if (rr >= pre && rr - pre < mine) {
        // block exclusive scan of the per-thread sums (the banned token's thread without it)
        const unsigned long long tsb = ts - ((ban >= t0 && ban < t1) ? wban : 0ull);
        unsigned long long inc = tsb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) s_rs[warp] = inc;
        __syncthreads();
        unsigned long long base = 0;
        for (int w = 0; w < warp; ++w) base += s_rs[w];
        const unsigned long long tpre = base + inc - tsb, r2 = rr - pre;
        if (r2 >= tpre && r2 - tpre < tsb) {
            // this thread's run: the first logit whose running sum passes r2
            const uint4* run = run_of(i);
            unsigned long long acc = tpre;
            int tok = -1;
            for (int k = 0; k < K && tok < 0 && t0 + k * VN < hi; ++k) {
                const int e0 = t0 + k * VN;
                float x[VN];
                LAZY_LOAD_VEC(i, run, k, x);
                unsigned long long w[VN];
#pragma unroll
                for (int j = 0; j < VN; ++j) w[j] = e0 + j != ban ? weight_of(x[j], m, c) : 0ull;
#pragma unroll
                for (int j = 0; j < VN; ++j) {
                    acc += w[j];
                    if (tok < 0 && acc > r2) tok = e0 + j;
                }
            }
            out[i] = tok;
        }
    } else if (rank == 0 && tid == 0 && rr >= Z) {
        out[i] = -1;                                 // nothing left to draw from
    }
    // rank 0 writes everything but the drawn position: the accepted drafts and the padding
    if (rank == 0) {
        if (tid == 0 && Z == 0) set_status(a.status, GDN_STATUS_EMPTY_DIST);
        for (int k = tid; k < RS; k += NT)
            if (k != i) out[k] = k < i ? dr[k] : -1;
        if (tid == 0) a.n_acc[b] = act == 1 ? i : N;
    }
    // a copy whose wait gave up may still be landing in this CTA's stages: wait once more
    if (tid == 0) {
        for (int q = 0; q < 2; ++q)
            if ((pending >> q) & 1u) (void)mbar_wait_bounded(&s_bar[q], (pend_par >> q) & 1u);
    }
}
#undef LAZY_LOAD_VEC

// Launch plan of the cluster path: cluster size CL, slice SL, vectors per thread K, threads NT.
struct LazyPlan {
    int CL, SL, K, NT;
    size_t smem;
};

static std::mutex g_plan_mu;
static std::map<std::tuple<unsigned long long, int, int, int, int>, LazyPlan> g_plans;

// The cluster path serves vocabularies of 8192 and more whose two-row slices fit shared memory;
// among the cluster sizes that fit, it takes the one with the fewest waves of clusters, weighing
// a wave as the row work of one CTA (1/CL) plus a fixed part (barriers, latency).
template <typename LT>
static bool lazy_plan(int V, int B, int N, LazyPlan* out) {
    if (V < 8192) return false;
    constexpr int VN = 16 / int(sizeof(LT));
    const unsigned long long ctx = current_context_id();
    const auto key = std::make_tuple(ctx, int(sizeof(LT)), V, B, N);
    std::lock_guard<std::mutex> lock(g_plan_mu);
    if (ctx) {
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            *out = it->second;
            return out->CL > 0;
        }
    }
    auto kern = accept_sample_lazy_kernel<LT>;
    constexpr size_t kMaxDyn = 225 * 1024;
    LazyPlan best{0, 0, 0, 0, 0};
    double best_cost = 1e300;
    int nsm = 0;
    if (device_sm_count(&nsm) == cudaSuccess && nsm > 0 &&
        smem_optin(reinterpret_cast<const void*>(kern), kMaxDyn) == cudaSuccess) {
        const bool big = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                              1) == cudaSuccess;
        (void)cudaGetLastError();
        for (int CL = big ? kMaxCL : 8; CL >= 1; --CL) {
            int SL = (V + CL - 1) / CL;
            SL = (SL + VN - 1) / VN * VN;
            const int nvec = SL / VN;
            int K = 1;
            while ((nvec + K - 1) / K > 1024) K += 2;
            int NT = ((nvec + K - 1) / K + 31) / 32 * 32;
            const size_t smem = size_t(2) * NT * K * 16 + (size_t(N) * 4 + 15) / 16 * 16;
            if (smem > kMaxDyn) continue;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = unsigned(CL);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(unsigned(CL));
            cfg.blockDim = dim3(unsigned(NT));
            cfg.dynamicSmemBytes = smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                (void)cudaGetLastError();
                continue;
            }
            // within one wave, CTAs beyond one per SM share SMs (a cluster waits for its slowest)
            const int waves = (B + n - 1) / n;
            const int per_sm = waves == 1 ? (B * CL + nsm - 1) / nsm : 1;
            const double cost = double(waves) * (double(per_sm) / CL + 0.25);
            if (cost < best_cost) {
                best_cost = cost;
                best = LazyPlan{CL, SL, K, NT, smem};
            }
        }
    }
    (void)cudaGetLastError();
    if (ctx) g_plans[key] = best;
    *out = best;
    return best.CL > 0;
}

template <typename LT>
static cudaError_t launch_lazy(const AcceptArgs& a, const LazyPlan& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.CL);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(a.B) * unsigned(p.CL));
    cfg.blockDim = dim3(unsigned(p.NT));
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, accept_sample_lazy_kernel<LT>, a, p.SL, p.K);
}

// ---------------------------------------------------------------- host launchers
void accept_chunking(int rows, int V, int* CH, int* CS) {
    int ch = rows > 0 ? (1216 + rows - 1) / rows : 1;
    ch = ch < 1 ? 1 : (ch > 64 ? 64 : ch);
    int cs = (V + ch - 1) / ch;
    cs = (cs + 7) / 8 * 8;
    if (cs < 8) cs = 8;
    *CS = cs;
    *CH = (V + cs - 1) / cs;
}

template <typename LT>
static cudaError_t greedy_t(const AcceptArgs& a, cudaStream_t s) {
    const unsigned rows = unsigned(a.B) * unsigned(a.N + 1);
    accept_rowmax_kernel<LT><<<dim3(rows, a.CH), kAccThreads, 0, s>>>(a);
    accept_greedy_scan_kernel<<<a.B, kAccThreads, (a.N + 1) * sizeof(int), s>>>(a);
    return cudaGetLastError();
}

template <typename LT>
static cudaError_t sample_t(const AcceptArgs& a, cudaStream_t s) {
    LazyPlan p;
    if (a.B <= 0x7fffffff / kMaxCL && a.N <= 4096 && lazy_plan<LT>(a.V, a.B, a.N, &p)) {
        const cudaError_t e = launch_lazy<LT>(a, p, s);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const unsigned rows = unsigned(a.B) * unsigned(a.N + 1);
    accept_rowmax_kernel<LT><<<dim3(rows, a.CH), kAccThreads, 0, s>>>(a);
    accept_weights_kernel<LT><<<dim3(rows, a.CH), kAccThreads, 0, s>>>(a);
    accept_sample_scan_kernel<LT><<<a.B, kAccThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename LT>
static cudaError_t tree_t(const AcceptArgs& a, cudaStream_t s) {
    const unsigned rows = unsigned(a.B) * unsigned(a.N + 1);
    accept_rowmax_kernel<LT><<<dim3(rows, a.CH), kAccThreads, 0, s>>>(a);
    accept_tree_scan_kernel<<<a.B, kAccThreads, (3 * a.N + 1) * sizeof(int), s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_accept_greedy(const AcceptArgs& a, int dtype, cudaStream_t s) {
    return dtype == GDN_DTYPE_BF16 ? greedy_t<__nv_bfloat16>(a, s) : greedy_t<float>(a, s);
}
cudaError_t launch_accept_sample(const AcceptArgs& a, int dtype, cudaStream_t s) {
    return dtype == GDN_DTYPE_BF16 ? sample_t<__nv_bfloat16>(a, s) : sample_t<float>(a, s);
}
cudaError_t launch_accept_tree(const AcceptArgs& a, int dtype, cudaStream_t s) {
    return dtype == GDN_DTYPE_BF16 ? tree_t<__nv_bfloat16>(a, s) : tree_t<float>(a, s);
}

}  // namespace gdn
