/*
 * oracle.h — declarations of the CPU oracle (test infrastructure only; see oracle.c).
 * Layouts follow the library's C ABI (dense row-major), with every floating-point tensor
 * widened to fp64 and logits given as fp32 (bf16 logits widen to fp32 exactly).
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct oracle_dims {
    int L, B, T, Hk, Hv, Dk, Dv, W, C;
    int act_silu;     /* 1: y = silu(conv(x)); 0: no activation (literal reading test mode) */
    int gate_dk;      /* 0: g [L][B][T][Hv]; 1: per-key-channel gates g [L][B][T][Hv][Dk] */
    double qk_scale;
    double l2_eps;
} oracle_dims;

/* qkv [L][B][T][C], conv_w [L][C][W], conv_state [L][B][W-1][C], g/beta [L][B][T][Hv] (g
 * [L][B][T][Hv][Dk] when gate_dk),
 * state [L][B][Hv][Dv][Dk] (row-major S: S(i,j) at [i][j]); out [L][B][T][Hv][Dv], tape_delta
 * same, tape_k [L][B][T][Hk][Dk]; node_state (optional) [L][B][T][Hv][Dv][Dk] = state after node.
 * parent [B][T] or NULL for a chain. */
void oracle_verify(const oracle_dims* dm, const int32_t* parent, const double* qkv,
                   const double* conv_w, const double* conv_state, const double* g,
                   const double* beta, const double* state, double* out, double* tape_delta,
                   double* tape_k, double* node_state);

/* Returns OR of 1 (n out of range) and 8 (bad path node); skips those sequences. */
int oracle_rollback(const oracle_dims* dm, const int32_t* path, int P, const int32_t* n_acc,
                    const double* tape_delta, const double* tape_k, const double* g,
                    const double* qkv, double* state, double* conv_state);

/* Threads for the loops over independent units (layers x sequences, sequences); 1 by default.
 * Results do not depend on it. */
void oracle_set_threads(int n);
int oracle_get_threads(void);
int oracle_openmp(void);

int oracle_argmax(const float* row, int V);
int oracle_accept_greedy(int B, int N, int V, int64_t row_stride, int64_t seq_stride,
                         const float* logits, const int32_t* drafts, int32_t* n_acc,
                         int32_t* out_tokens);

float oracle_exp2_spec(float x);
float oracle_scale_c(float temperature);
uint64_t oracle_weights(const float* row, int V, float c, int ban, uint64_t* w);
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]);
uint64_t oracle_draw(uint64_t seed, uint32_t round, uint32_t seq, uint32_t row, uint32_t purpose,
                     uint64_t Z);
int oracle_accept_sample(int B, int N, int V, int64_t row_stride, int64_t seq_stride,
                         const float* logits, const int32_t* drafts, float temperature,
                         uint64_t seed, uint64_t round, int32_t* n_acc, int32_t* out_tokens);

int oracle_accept_tree(int B, int T, int V, int64_t row_stride, int64_t seq_stride,
                       const float* logits, const int32_t* parent, const int32_t* tokens, int P,
                       int32_t* path, int32_t* n_acc, int32_t* out_tokens);

/* Full-attention layer verify and KV truncation (see oracle.c). q, out [L][B][T][Hq][D];
 * k_new, v_new [L][B][T][Hkv][D]; k_cache, v_cache [L][B][Hkv][ctx][D] (token-major, appended in
 * place); kv_len [B]. Returns 1 if some kv_len[b] is outside [0, ctx - T] (sequence skipped). */
typedef struct oracle_attn_dims {
    int L, B, T, Hq, Hkv, D, ctx;
    double scale;
} oracle_attn_dims;

int oracle_attn_verify(const oracle_attn_dims* a, const int32_t* kv_len, const double* q,
                       const double* k_new, const double* v_new, double* k_cache,
                       double* v_cache, double* out);

/* kv_len[b] += n_acc[b] for n in [0, T]; returns 1 (and skips b) for any other n. */
int oracle_attn_truncate(int B, int T, const int32_t* n_acc, int32_t* kv_len);

#ifdef __cplusplus
}
#endif

#endif
