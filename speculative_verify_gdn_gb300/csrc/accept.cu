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
// zero for n < -64. p lies in [2^-1/2, 2^1/2] (a normal fp32 with 24-bit significand M, exponent
// E), and p · 2^n · 2^32 is exact in fp32, so w = floor(M · 2^(E + n + 9)): a shift, no float to
// 64-bit conversion. n comes from the bits of x + 1.5·2^23 (round to nearest even, exact for
// |x| < 2^22).
// A NaN logit counts as −∞ (weight 0; the row max never is NaN, the argmax pass skips NaN), and so
// does a NaN x from a −∞ or NaN logit against a −∞ maximum.
__device__ __forceinline__ unsigned long long weight_of(float l, float m, float c) {
    const float x = __fmul_rn(__fsub_rn(l, m), c);
    if (!(x >= -100.0f)) return 0ull;                   // rint(x) < -64 as well, or x NaN
    const float t = __fadd_rn(x, 12582912.0f);
    const int n = __float_as_int(t) - 0x4B400000;       // rint(x)
    if (n < -64) return 0ull;
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
    const unsigned long long M = (pb & 0x7FFFFFu) | 0x800000u;
    const int sh = int(pb >> 23) - 127 + n + 9;
    return sh >= 0 ? (M << sh) : (M >> (-sh));
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
    extern __shared__ int s_am[];   // [T + 1]
    __shared__ int s_bad;
    const int b = blockIdx.x, T = a.N, RS = T + 1, P = a.P;
    const int32_t* par = a.parent + size_t(b) * T;
    const int32_t* tok = a.drafts + size_t(b) * T;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < RS; i += kAccThreads) {
        s_am[i] = key_index(row_best_key(a, b * RS + i));
        if (i < T) {
            if (par[i] < -1 || par[i] >= i) atomicOr(&s_bad, 1);
            if (tok[i] < 0 || tok[i] >= a.V) atomicOr(&s_bad, 2);
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
    accept_tree_scan_kernel<<<a.B, kAccThreads, (a.N + 1) * sizeof(int), s>>>(a);
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
