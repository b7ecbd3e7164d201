/*
 * oracle.c — plain, slow, obviously-correct CPU oracle for speculative verify / accept / rollback
 * on GatedDeltaNet layers. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
 * CPU-baseline leg may call it; the library never does. It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Floating point is fp64 (the pages fix no precision), evaluated with contraction disabled
 * (built with -ffp-contract=off) so the same expression always rounds the same way. The sampling
 * decision is the exception: the integer-weight contract fixes fp32 for the weights, and both
 * sides take that decision in fp32 (see oracle_exp2_spec).
 *
 * Sources (page titles):
 *  [GDN]  "Speculative Decoding on GDN Hybrid Architectures: A 31-Experiment Investigation":
 *         §2.1 GDN layer = Conv1D state + gated delta state, sequential per token;
 *         §2.2 multi-token verification; §3.3 experiment 7 (snapshot / restore / replay);
 *         §4 "Tape-Replay 回滚": tape of δ [B,T,Hv,Dv], k [B,T,Hk,Dk], g [B,T,Hv] and raw qkv;
 *         restore the snapshot, replay state = state*g[t] + k[t]*tape[t] for t < n accepted;
 *         conv state rebuilt from the last (conv_kernel_size − 1) raw qkv rows.
 *  [XS]   "Phase 25: 三种投机解码方法对比 (Small Model / EAGLE / MTP)", §2 algorithm: accept the
 *         longest prefix with draft == argmax, then append the target's argmax as correction.
 *  [COL]  colibrì analysis ch.08 "MTP 投机解码与预取", §5 rejection sampling: accept draft k with
 *         probability p(draft k); on rejection ban that token, zero it, renormalise, resample.
 *  [GDN] §2.1 / §2.2 also fix the hybrid's other layer type: standard multi-head attention with a
 *         KV cache, whose N verify positions are computed in parallel (oracle_attn_verify), and
 *         whose rejected positions are dropped by truncating the cache length (oracle_attn_truncate).
 * The update rule itself is the standard gated delta rule
 *     S_t = g_t S_{t-1} (I − β_t k_t k_tᵀ) + β_t v_t k_tᵀ,  o_t = S_t q_t,
 * written here in its innovation form u = g_t S k_t, δ_t = β_t (v_t − u), S ← g_t S + δ_t k_tᵀ,
 * which is exactly the form the [GDN] §4 replay rule replays.
 *
 * Parity pins cover every function below; none is unpinned: tests/test_oracle_pins.py (verify,
 * rollback, accept, the sampling contract), tests/test_gate_dk.py (per-key-channel gates),
 * tests/test_attn_oracle.py (attention verify and truncation).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------
 * Threads. Layers, sequences and value heads are independent units of verify and rollback, and
 * sequences of accept ([GDN] §2.2: verification is per sequence; the state is per layer and head),
 * so with more than one thread the loops over them are split between OpenMP threads, each with
 * its own scratch. Every unit is still computed by one thread with the same expressions in the
 * same order: the results are bit-identical to the single-threaded run (a CPU test checks it).
 * ------------------------------------------------------------------------------------------ */
static int g_threads = 1;

void oracle_set_threads(int n) { g_threads = n < 1 ? 1 : n; }
int oracle_get_threads(void) { return g_threads; }
/* 1 when built with OpenMP (else the thread count has no effect) */
int oracle_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* ------------------------------------------------------------------------------------------
 * Indexing helpers. Layouts are those of the C ABI, dense row-major.
 * ------------------------------------------------------------------------------------------ */
#define IDX2(a, b, nb) ((size_t)(a) * (size_t)(nb) + (size_t)(b))

static double silu(double y) { return y / (1.0 + exp(-y)); }

/* Raw input row of the conv window of node v at distance d (d = 0 is v itself) for one channel.
 * anc[0..depth-1] = v, parent(v), parent(parent(v)), ...  Beyond the root the window continues
 * into the conv state, newest row last: distance depth maps to conv_state row W-2.           */
static double window_value(const double* qkv_lb, const double* cs_lb, int C, int W,
                           const int* anc, int depth, int d, int c) {
    if (d < depth) return qkv_lb[IDX2(anc[d], c, C)];
    int e = d - depth;           /* 0 = newest conv-state row */
    int row = W - 2 - e;
    return cs_lb[IDX2(row, c, C)];
}

/* ------------------------------------------------------------------------------------------
 * Verify (chain when parent == NULL, tree otherwise).
 * ------------------------------------------------------------------------------------------ */
void oracle_verify(const oracle_dims* dm, const int32_t* parent, const double* qkv,
                   const double* conv_w, const double* conv_state, const double* g,
                   const double* beta, const double* state, double* out, double* tape_delta,
                   double* tape_k, double* node_state) {
    const int L = dm->L, B = dm->B, T = dm->T, Hk = dm->Hk, Hv = dm->Hv, Dk = dm->Dk,
              Dv = dm->Dv, W = dm->W, C = dm->C;
    const int qoff = 0, koff = Hk * Dk, voff = 2 * Hk * Dk;
    const int group = Hv / Hk;

#pragma omp parallel num_threads(g_threads) if (g_threads > 1)
    {
    double* y = (double*)malloc(sizeof(double) * (size_t)T * C);   /* conv+act output */
    int* anc = (int*)malloc(sizeof(int) * (size_t)(T + 1));
    double* S_nodes = (double*)malloc(sizeof(double) * (size_t)T * Dv * Dk); /* S per node */
    double* Sp = (double*)malloc(sizeof(double) * (size_t)Dv * Dk);

#pragma omp for collapse(2) schedule(dynamic)
    for (int l = 0; l < L; ++l) {
        for (int b = 0; b < B; ++b) {
            const size_t lb = (size_t)l * B + b;
            const double* qkv_lb = qkv + lb * (size_t)T * C;
            const double* cs_lb = conv_state + lb * (size_t)(W - 1) * C;
            const double* w_l = conv_w + (size_t)l * C * W;
            const int32_t* par = parent ? parent + (size_t)b * T : NULL;

            /* (1) causal depthwise conv over each node's window, then the activation */
            for (int v = 0; v < T; ++v) {
                int depth = 0, a = v;
                while (a >= 0) { anc[depth++] = a; a = par ? par[a] : a - 1; }
                for (int c = 0; c < C; ++c) {
                    double acc = 0.0;
                    for (int j = 0; j < W; ++j) {
                        /* tap W-1 multiplies the current token (distance 0) */
                        double x = window_value(qkv_lb, cs_lb, C, W, anc, depth, W - 1 - j, c);
                        acc = acc + w_l[IDX2(c, j, W)] * x;
                    }
                    y[IDX2(v, c, C)] = dm->act_silu ? silu(acc) : acc;
                }
            }
            /* (2) split into heads and L2-normalise q and k per head */
            for (int v = 0; v < T; ++v) {
                for (int hk = 0; hk < Hk; ++hk) {
                    double* q = y + IDX2(v, qoff + hk * Dk, C);
                    double* k = y + IDX2(v, koff + hk * Dk, C);
                    double sq = 0.0, sk = 0.0;
                    for (int j = 0; j < Dk; ++j) { sq += q[j] * q[j]; sk += k[j] * k[j]; }
                    double iq = 1.0 / sqrt(sq + dm->l2_eps), ik = 1.0 / sqrt(sk + dm->l2_eps);
                    for (int j = 0; j < Dk; ++j) { q[j] = q[j] * iq; k[j] = k[j] * ik; }
                    for (int j = 0; j < Dk; ++j)
                        tape_k[(((lb * T + v) * Hk) + hk) * (size_t)Dk + j] = k[j];
                }
            }
            /* (3) gated delta recurrence per value head, node by node from the parent's state */
            for (int h = 0; h < Hv; ++h) {
                const int hk = h / group;
                const double* S0 = state + (lb * Hv + h) * (size_t)Dv * Dk; /* [i][j] */
                for (int v = 0; v < T; ++v) {
                    int p = par ? par[v] : v - 1;
                    /* parent state S_p as a plain row-major Dv x Dk matrix */
                    for (int i = 0; i < Dv; ++i)
                        for (int j = 0; j < Dk; ++j)
                            Sp[IDX2(i, j, Dk)] = (p < 0) ? S0[IDX2(i, j, Dk)]
                                                         : S_nodes[((size_t)p * Dv + i) * Dk + j];
                    const double* k = y + IDX2(v, koff + hk * Dk, C);
                    const double* q = y + IDX2(v, qoff + hk * Dk, C);
                    const double* vv = y + IDX2(v, voff + h * Dv, C);
                    const double bv = beta[(lb * T + v) * Hv + h];
                    double* Sv = S_nodes + (size_t)v * Dv * Dk;
                    if (!dm->gate_dk) {
                        const double gv = g[(lb * T + v) * Hv + h];
                        for (int i = 0; i < Dv; ++i) {
                            double sk = 0.0;
                            for (int j = 0; j < Dk; ++j) sk += Sp[IDX2(i, j, Dk)] * k[j];
                            double u = gv * sk;
                            double delta = bv * (vv[i] - u);
                            tape_delta[(((lb * T + v) * Hv) + h) * (size_t)Dv + i] = delta;
                            for (int j = 0; j < Dk; ++j)
                                Sv[IDX2(i, j, Dk)] = gv * Sp[IDX2(i, j, Dk)] + delta * k[j];
                        }
                    } else {
                        /* per-key-channel gate a_j ([GDN] §4 tape layout [B, T, Hv, Dk]): the
                         * decayed state S_p diag(a) takes the place of g S_p */
                        const double* av = g + ((lb * T + v) * Hv + h) * (size_t)Dk;
                        for (int i = 0; i < Dv; ++i) {
                            double u = 0.0;
                            for (int j = 0; j < Dk; ++j) u += (av[j] * Sp[IDX2(i, j, Dk)]) * k[j];
                            double delta = bv * (vv[i] - u);
                            tape_delta[(((lb * T + v) * Hv) + h) * (size_t)Dv + i] = delta;
                            for (int j = 0; j < Dk; ++j)
                                Sv[IDX2(i, j, Dk)] = av[j] * Sp[IDX2(i, j, Dk)] + delta * k[j];
                        }
                    }
                    for (int i = 0; i < Dv; ++i) {
                        double o = 0.0;
                        for (int j = 0; j < Dk; ++j) o += Sv[IDX2(i, j, Dk)] * q[j];
                        out[(((lb * T + v) * Hv) + h) * (size_t)Dv + i] = dm->qk_scale * o;
                    }
                    if (node_state) {
                        double* dst = node_state + ((lb * T + v) * Hv + h) * (size_t)Dv * Dk;
                        for (int i = 0; i < Dv; ++i)
                            for (int j = 0; j < Dk; ++j) dst[IDX2(i, j, Dk)] = Sv[IDX2(i, j, Dk)];
                    }
                }
            }
        }
    }
    free(Sp);
    free(S_nodes);
    free(anc);
    free(y);
    }
}

/* ------------------------------------------------------------------------------------------
 * Rollback by tape replay ([GDN] §4). Chain when path == NULL, else along path[b][0..n-1].
 * ------------------------------------------------------------------------------------------ */
int oracle_rollback(const oracle_dims* dm, const int32_t* path, int P, const int32_t* n_acc,
                    const double* tape_delta, const double* tape_k, const double* g,
                    const double* qkv, double* state, double* conv_state) {
    const int L = dm->L, B = dm->B, T = dm->T, Hk = dm->Hk, Hv = dm->Hv, Dk = dm->Dk,
              Dv = dm->Dv, W = dm->W, C = dm->C;
    const int group = Hv / Hk;
    int bad = 0;
#pragma omp parallel num_threads(g_threads) if (g_threads > 1) reduction(| : bad)
    {
    int* nodes = (int*)malloc(sizeof(int) * (size_t)(T + 1));
    double* rows = (double*)malloc(sizeof(double) * (size_t)(W - 1 + T + 1));
#pragma omp for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        int n = n_acc[b];
        int cap = path ? P : T;
        if (n < 0 || n > cap || n > T) { bad |= 1; continue; }
        if (n == 0) continue;            /* the snapshot is still in place */
        int ok = 1;
        for (int s = 0; s < n; ++s) {
            nodes[s] = path ? path[(size_t)b * P + s] : s;
            if (nodes[s] < 0 || nodes[s] >= T) ok = 0;
        }
        if (!ok) { bad |= 8; continue; }
        for (int l = 0; l < L; ++l) {
            const size_t lb = (size_t)l * B + b;
            for (int h = 0; h < Hv; ++h) {
                const int hk = h / group;
                double* S = state + (lb * Hv + h) * (size_t)Dv * Dk; /* [i][j] */
                for (int s = 0; s < n; ++s) {
                    const int t = nodes[s];
                    const double* dl = tape_delta + ((lb * T + t) * Hv + h) * (size_t)Dv;
                    const double* kt = tape_k + ((lb * T + t) * Hk + hk) * (size_t)Dk;
                    /* state = state * g[t] + k[t] * tape[t], elementwise S(i,j); g[t] is one
                     * value per head, or one per key channel j */
                    if (!dm->gate_dk) {
                        const double gt = g[(lb * T + t) * Hv + h];
                        for (int i = 0; i < Dv; ++i)
                            for (int j = 0; j < Dk; ++j)
                                S[IDX2(i, j, Dk)] = gt * S[IDX2(i, j, Dk)] + dl[i] * kt[j];
                    } else {
                        const double* at = g + ((lb * T + t) * Hv + h) * (size_t)Dk;
                        for (int i = 0; i < Dv; ++i)
                            for (int j = 0; j < Dk; ++j)
                                S[IDX2(i, j, Dk)] = at[j] * S[IDX2(i, j, Dk)] + dl[i] * kt[j];
                    }
                }
            }
            /* conv state: last W-1 raw rows of (conv_state ++ accepted qkv rows) */
            double* cs = conv_state + lb * (size_t)(W - 1) * C;
            const double* x = qkv + lb * (size_t)T * C;
            for (int c = 0; c < C; ++c) {
                int m = 0;
                for (int r = 0; r < W - 1; ++r) rows[m++] = cs[IDX2(r, c, C)];
                for (int s = 0; s < n; ++s) rows[m++] = x[IDX2(nodes[s], c, C)];
                for (int r = 0; r < W - 1; ++r) cs[IDX2(r, c, C)] = rows[m - (W - 1) + r];
            }
        }
    }
    free(rows);
    free(nodes);
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------
 * Greedy acceptance ([XS] §2 algorithm; [COL] §5 greedy path). Row i judges draft i; row N is
 * the bonus row. argmax returns the lowest index among equal maxima.
 * ------------------------------------------------------------------------------------------ */
/* A NaN logit counts as −∞: it is never the maximum unless every entry is NaN or −∞, and then
 * the lowest index (0) is returned, like any tie. */
static float logit_or_neg_inf(float x) { return isnan(x) ? -INFINITY : x; }

int oracle_argmax(const float* row, int V) {
    int best = 0;
    float m = logit_or_neg_inf(row[0]);
    for (int v = 1; v < V; ++v)
        if (logit_or_neg_inf(row[v]) > m) { best = v; m = logit_or_neg_inf(row[v]); }
    return best;
}

int oracle_accept_greedy(int B, int N, int V, int64_t row_stride, int64_t seq_stride,
                         const float* logits, const int32_t* drafts, int32_t* n_acc,
                         int32_t* out_tokens) {
    int bad = 0;
#pragma omp parallel for num_threads(g_threads) if (g_threads > 1) reduction(| : bad) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        const float* lg = logits + (size_t)b * seq_stride;
        const int32_t* dr = drafts + (size_t)b * N;
        int32_t* out = out_tokens + (size_t)b * (N + 1);
        for (int i = 0; i <= N; ++i) out[i] = -1;
        int okd = 1;
        for (int i = 0; i < N; ++i)
            if (dr[i] < 0 || dr[i] >= V) okd = 0;
        if (!okd) { bad |= 4; n_acc[b] = 0; continue; }
        int accepted = 0;
        while (accepted < N && dr[accepted] == oracle_argmax(lg + (size_t)accepted * row_stride, V))
            accepted += 1;
        int correction = oracle_argmax(lg + (size_t)accepted * row_stride, V);
        for (int i = 0; i < accepted; ++i) out[i] = dr[i];
        out[accepted] = correction;
        n_acc[b] = accepted;
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------
 * Integer-weight sampling contract.
 *
 * exp2 by Cody–Waite range reduction (W. J. Cody and W. Waite, "Software Manual for the
 * Elementary Functions", 1980): x = n + f with n = nearest integer (ties to even), f in
 * [-1/2, 1/2]; 2^f by its Taylor series to degree 7, coefficients (ln 2)^k / k! rounded to fp32,
 * evaluated by Horner with fused multiply-adds; then an exact scaling by 2^n. Everything in fp32.
 * ------------------------------------------------------------------------------------------ */
/* (ln 2)^k / k!, computed in double and rounded once to fp32 */
static float g_coef[8];
static int g_coef_ready = 0;

static void init_coefs(void) {
    double c = 1.0;
    for (int k = 0; k < 8; ++k) {
        if (k > 0) c = c * log(2.0) / (double)k;
        g_coef[k] = (float)c;
    }
    g_coef_ready = 1;
}

float oracle_exp2_spec(float x) {
    if (!g_coef_ready) init_coefs();
    float n = rintf(x);                    /* round to nearest, ties to even */
    if (!(n >= -64.0f)) return 0.0f;       /* 2^x < 2^-63.5, or x NaN (a NaN or −∞ logit
                                              against a −∞ maximum): weight 0 */
    float f = x - n;                       /* exact */
    float p = g_coef[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, f, g_coef[k]);
    return ldexpf(p, (int)n);              /* exact: result stays a normal float */
}

float oracle_scale_c(float temperature) {
    return (float)((1.0 / log(2.0)) / (double)temperature);
}

/* weights of one row; ban < 0 for none. Returns Z = Σ w. */
uint64_t oracle_weights(const float* row, int V, float c, int ban, uint64_t* w) {
    /* NaN logits count as −∞ (weight 0), as in oracle_argmax */
    float m = logit_or_neg_inf(row[0]);
    for (int v = 1; v < V; ++v)
        if (logit_or_neg_inf(row[v]) > m) m = logit_or_neg_inf(row[v]);
    uint64_t Z = 0;
    for (int v = 0; v < V; ++v) {
        float dlt = logit_or_neg_inf(row[v]) - m;
        float x = dlt * c;
        float e = oracle_exp2_spec(x);
        uint64_t wv = (uint64_t)(e * 4294967296.0f);   /* e * 2^32 is exact; truncation = floor */
        if (v == ban) wv = 0;
        w[v] = wv;
        Z += wv;
    }
    return Z;
}

/* Philox4x32-10 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random numbers:
 * as easy as 1, 2, 3", SC'11): 10 rounds of two 32x32->64 multiplies with the Weyl key schedule. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* r = floor(U * Z / 2^128), U = (x3:x2:x1:x0) the 128-bit Philox output, by exact integer math */
uint64_t oracle_draw(uint64_t seed, uint32_t round, uint32_t seq, uint32_t row, uint32_t purpose,
                     uint64_t Z) {
    uint32_t ctr[4] = {round, seq, row, purpose};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    oracle_philox4x32_10(ctr, key, x);
    unsigned __int128 U = ((unsigned __int128)x[3] << 96) | ((unsigned __int128)x[2] << 64) |
                          ((unsigned __int128)x[1] << 32) | (unsigned __int128)x[0];
    /* U*Z < 2^179: split U into 64-bit halves to stay within 128-bit arithmetic */
    uint64_t Uh = (uint64_t)(U >> 64), Ul = (uint64_t)U;
    unsigned __int128 hi = (unsigned __int128)Uh * Z;
    unsigned __int128 lo = (unsigned __int128)Ul * Z;
    unsigned __int128 sum = hi + (lo >> 64);
    return (uint64_t)(sum >> 64);
}

static int pick_by_weight(const uint64_t* w, int V, uint64_t r) {
    uint64_t acc = 0;
    for (int v = 0; v < V; ++v) {
        acc += w[v];
        if (acc > r) return v;
    }
    return -1;
}

int oracle_accept_sample(int B, int N, int V, int64_t row_stride, int64_t seq_stride,
                         const float* logits, const int32_t* drafts, float temperature,
                         uint64_t seed, uint64_t round, int32_t* n_acc, int32_t* out_tokens) {
    if (!(temperature > 0.0f))
        return oracle_accept_greedy(B, N, V, row_stride, seq_stride, logits, drafts, n_acc,
                                    out_tokens);
    int bad = 0;
    if (!g_coef_ready) init_coefs();     /* before the threads share the table */
    const float c = oracle_scale_c(temperature);
    const uint32_t rnd = (uint32_t)round;
#pragma omp parallel num_threads(g_threads) if (g_threads > 1) reduction(| : bad)
    {
    uint64_t* w = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
#pragma omp for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        const float* lg = logits + (size_t)b * seq_stride;
        const int32_t* dr = drafts + (size_t)b * N;
        int32_t* out = out_tokens + (size_t)b * (N + 1);
        for (int i = 0; i <= N; ++i) out[i] = -1;
        int okd = 1;
        for (int i = 0; i < N; ++i)
            if (dr[i] < 0 || dr[i] >= V) okd = 0;
        if (!okd) { bad |= 4; n_acc[b] = 0; continue; }
        int n = N;
        for (int i = 0; i < N; ++i) {
            const float* row = lg + (size_t)i * row_stride;
            uint64_t Z = oracle_weights(row, V, c, -1, w);
            uint64_t r = oracle_draw(seed, rnd, (uint32_t)b, (uint32_t)i, 0u, Z);
            if (r < w[dr[i]]) { out[i] = dr[i]; continue; }       /* accept w.p. p(draft) */
            /* reject: ban the draft, renormalise, resample from the rest */
            uint64_t Zb = Z - w[dr[i]];
            w[dr[i]] = 0;
            uint64_t r2 = oracle_draw(seed, rnd, (uint32_t)b, (uint32_t)i, 1u, Zb);
            out[i] = pick_by_weight(w, V, r2);
            n = i;
            break;
        }
        if (n == N) {   /* all accepted: the bonus token from row N */
            const float* row = lg + (size_t)N * row_stride;
            uint64_t Z = oracle_weights(row, V, c, -1, w);
            uint64_t r2 = oracle_draw(seed, rnd, (uint32_t)b, (uint32_t)N, 1u, Z);
            out[N] = pick_by_weight(w, V, r2);
        }
        n_acc[b] = n;
    }
    free(w);
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------
 * Greedy tree acceptance: longest matching root-to-leaf path. Row 0 judges the children of the
 * committed context; row 1+v judges the children of node v.
 * ------------------------------------------------------------------------------------------ */
int oracle_accept_tree(int B, int T, int V, int64_t row_stride, int64_t seq_stride,
                       const float* logits, const int32_t* parent, const int32_t* tokens, int P,
                       int32_t* path, int32_t* n_acc, int32_t* out_tokens) {
    int bad = 0;
#pragma omp parallel for num_threads(g_threads) if (g_threads > 1) reduction(| : bad) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        const float* lg = logits + (size_t)b * seq_stride;
        const int32_t* par = parent + (size_t)b * T;
        const int32_t* tok = tokens + (size_t)b * T;
        int32_t* pth = path + (size_t)b * P;
        int32_t* out = out_tokens + (size_t)b * (P + 1);
        for (int i = 0; i < P; ++i) pth[i] = -1;
        for (int i = 0; i <= P; ++i) out[i] = -1;
        int okp = 1, okt = 1;
        for (int v = 0; v < T; ++v) {
            if (par[v] < -1 || par[v] >= v) okp = 0;
            if (tok[v] < 0 || tok[v] >= V) okt = 0;
        }
        if (!okp || !okt) { bad |= (okp ? 0 : 2) | (okt ? 0 : 4); n_acc[b] = 0; continue; }
        int cur = -1, n = 0;
        int am = oracle_argmax(lg, V);
        while (n < P) {
            int next = -1;
            for (int v = 0; v < T; ++v)
                if (par[v] == cur && tok[v] == am) { next = v; break; }
            if (next < 0) break;
            pth[n] = next;
            out[n] = tok[next];
            n += 1;
            cur = next;
            am = oracle_argmax(lg + (size_t)(1 + cur) * row_stride, V);
        }
        out[n] = am;
        n_acc[b] = n;
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------
 * Full-attention layer verify ([GDN] §2.1: the hybrid's attention layers are standard multi-head
 * attention over a KV cache; §2.2: the N verify positions run in parallel, not step by step).
 * Per layer l and sequence b with n0 = kv_len[b] committed rows: the T new key / value rows are
 * written to cache rows n0 .. n0+T-1 of their kv head; then query row (i, hq) reads kv head
 * hq / (Hq / Hkv) and attends causally to rows 0 .. n0+i:
 *     s_j = scale · q·k_j,   p = softmax(s),   o = Σ_j p_j v_j.
 * The softmax is evaluated as exp(s_j − max s) / Σ exp(s_j − max s) (the same quotient).
 * ------------------------------------------------------------------------------------------ */
int oracle_attn_verify(const oracle_attn_dims* a, const int32_t* kv_len, const double* q,
                       const double* k_new, const double* v_new, double* k_cache,
                       double* v_cache, double* out) {
    const int L = a->L, B = a->B, T = a->T, Hq = a->Hq, Hkv = a->Hkv, D = a->D, ctx = a->ctx;
    const int group = Hq / Hkv;
    int bad = 0;
    double* s = (double*)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
    for (int b = 0; b < B; ++b) {
        const int n0 = kv_len[b];
        if (n0 < 0 || n0 > ctx - T) { bad |= 1; continue; }
        for (int l = 0; l < L; ++l) {
            const size_t lb = (size_t)l * B + b;
            /* append the T new rows */
            for (int i = 0; i < T; ++i)
                for (int h = 0; h < Hkv; ++h) {
                    const size_t src = ((lb * T + i) * Hkv + h) * (size_t)D;
                    const size_t dst = ((lb * Hkv + h) * (size_t)ctx + (size_t)(n0 + i)) * D;
                    for (int e = 0; e < D; ++e) {
                        k_cache[dst + e] = k_new[src + e];
                        v_cache[dst + e] = v_new[src + e];
                    }
                }
            /* causal attention of every query row */
            for (int i = 0; i < T; ++i)
                for (int hq = 0; hq < Hq; ++hq) {
                    const int h = hq / group;
                    const double* qv = q + ((lb * T + i) * Hq + hq) * (size_t)D;
                    const double* K = k_cache + (lb * Hkv + h) * (size_t)ctx * D;
                    const double* V = v_cache + (lb * Hkv + h) * (size_t)ctx * D;
                    const int n = n0 + i + 1;          /* visible rows 0 .. n0+i */
                    double m = -INFINITY;
                    for (int j = 0; j < n; ++j) {
                        double dot = 0.0;
                        for (int e = 0; e < D; ++e) dot += qv[e] * K[(size_t)j * D + e];
                        s[j] = a->scale * dot;
                        if (s[j] > m) m = s[j];
                    }
                    double z = 0.0;
                    for (int j = 0; j < n; ++j) {
                        s[j] = exp(s[j] - m);
                        z += s[j];
                    }
                    double* o = out + ((lb * T + i) * Hq + hq) * (size_t)D;
                    for (int e = 0; e < D; ++e) {
                        double acc = 0.0;
                        for (int j = 0; j < n; ++j) acc += s[j] * V[(size_t)j * D + e];
                        o[e] = acc / z;
                    }
                }
        }
    }
    free(s);
    return bad;
}

/* KV truncation on reject: of the T appended rows the first n (the accepted drafts) stay, the
 * rest are dropped by the length alone (their slots are overwritten next round). */
int oracle_attn_truncate(int B, int T, const int32_t* n_acc, int32_t* kv_len) {
    int bad = 0;
    for (int b = 0; b < B; ++b) {
        const int n = n_acc[b];
        if (n < 0 || n > T) { bad |= 1; continue; }
        kv_len[b] += n;
    }
    return bad;
}

