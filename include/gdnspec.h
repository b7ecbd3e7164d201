/*
 * gdnspec.h — C ABI of the GB300 speculative-verify path for GatedDeltaNet (GDN) layers.
 *
 * One speculative round on the GDN layers of a hybrid model is three calls:
 *
 *   gdn_verify    run T draft positions through the GDN layers: causal depthwise conv + SiLU,
 *                 L2-normalised q/k, the gated delta rule, per-position outputs, and an
 *                 innovation tape. The recurrent state and the conv state are READ ONLY, so the
 *                 pre-verify snapshot stays in place.
 *   spec_accept   decide how many drafts to keep from the verify logits: greedy longest-prefix
 *                 argmax match, or Leviathan rejection sampling with point-mass drafts.
 *   gdn_rollback  commit the accepted prefix: restore-from-snapshot (implicit: the state was never
 *                 written) and replay only the accepted steps from the tape, O(n_accepted); rebuild
 *                 the conv state from the raw qkv rows.
 *
 * Tree variants (gdn_verify_tree, spec_accept_tree, gdn_rollback_path) walk a draft token tree
 * instead of a chain.
 *
 * Sources. "GDN investigation" below is the write-up "Speculative Decoding on GDN Hybrid
 * Architectures: A 31-Experiment Investigation"; "xserv docs/25" is "Phase 25: 三种投机解码方法对比
 * (Small Model / EAGLE / MTP)"; "colibrì ch.08" is the colibrì analysis chapter "MTP 投机解码与预取".
 *
 * Conventions common to every call.
 *  - Ownership: the caller owns every buffer. No call allocates, frees or synchronises.
 *  - Device pointers unless stated. Every call enqueues on `stream` and returns at once.
 *  - Layouts are dense row-major in the order written, e.g. [L][B][T][C] means
 *    element (l,b,t,c) lives at ((l*B + b)*T + t)*C + c.
 *  - Return value: GDN_OK, or an error code with a message in gdn_last_error(). On a non-OK
 *    return nothing was enqueued. Host-side argument checks never touch the GPU.
 *  - `status` (optional, may be NULL): one device uint32_t. Kernels OR GDN_STATUS_* bits into it
 *    when they meet an out-of-range device value (an accepted count, a parent index, a token);
 *    the offending unit is skipped. Kernels never trap. Read it after synchronising the stream;
 *    gdn_status_check() maps a non-zero word to GDN_ERR_DEVICE_STATUS with a readable message.
 *  - GDN_STATUS_WAIT_TIMEOUT means a bounded on-chip wait gave up (every mbarrier / copy wait in
 *    the kernels is limited to about one second of wall time instead of spinning forever). After
 *    it, every output of that call — of every unit, not only the one that timed out — is
 *    undefined and must be discarded: a unit that gave up may have left a copy in flight into
 *    shared memory that a later unit on the same SM then reuses.
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ---------------------------------------------------------------------- */
#define GDN_OK                0
#define GDN_ERR_INVALID_ARG   1  /* null pointer, negative or inconsistent size, misalignment */
#define GDN_ERR_UNSUPPORTED   2  /* valid but not built: head dims, T, W outside the kernel set */
#define GDN_ERR_CUDA          3  /* a CUDA launch or attribute call failed (message has the name) */
#define GDN_ERR_DEVICE_STATUS 4  /* gdn_status_check: the kernels reported a device-side problem */

/* ---- device status bits (OR-ed into *status by the kernels) ----------------------------- */
#define GDN_STATUS_BAD_NACC    0x1u  /* rollback: accepted count outside [0, T] */
#define GDN_STATUS_BAD_PARENT  0x2u  /* tree: parent not in [-1, v) for node v */
#define GDN_STATUS_BAD_TOKEN   0x4u  /* accept: draft / tree token outside [0, V) */
#define GDN_STATUS_BAD_PATH    0x8u  /* path rollback: path node out of range */
#define GDN_STATUS_EMPTY_DIST  0x10u /* sampling: a distribution with zero total weight */
#define GDN_STATUS_WAIT_TIMEOUT 0x20u /* a bounded on-chip wait gave up (results unspecified) */
#define GDN_STATUS_BAD_LEN     0x40u /* attention: kv_len outside [0, ctx - T] (or length overflow) */

/* ---- element types ---------------------------------------------------------------------- */
#define GDN_DTYPE_F32   0
#define GDN_DTYPE_BF16  1

/* ---- accept modes ----------------------------------------------------------------------- */
#define SPEC_MODE_GREEDY  0
#define SPEC_MODE_SAMPLE  1

/*
 * Shapes of one gdn_verify / gdn_rollback call.
 *  L   layers covered by the call (each layer has its own inputs, weights and state slices)
 *  B   sequences
 *  T   verify positions per sequence (chain: the N drafts; tree: the node count)
 *  Hk, Hv  key heads and value heads, Hv a multiple of Hk; value head h reads key head
 *          h / (Hv/Hk) (consecutive grouping)
 *  Dk, Dv  head dims; the kernels are built for Dk == Dv in {32, 64, 128}
 *  W   conv width, 1..4
 *  C   qkv channels; must equal 2*Hk*Dk + Hv*Dv, ordered [q | k | v], each head-major
 *  io_dtype  GDN_DTYPE_BF16 or GDN_DTYPE_F32 for qkv, conv_w, conv_state and out
 *  qk_scale  multiplies the output o_t (1.0 for the plain o_t = S_t q_t)
 *  l2_eps    x / sqrt(sum x^2 + l2_eps) normalises q and k (1e-6)
 */
typedef struct gdn_dims {
    int32_t L, B, T;
    int32_t Hk, Hv, Dk, Dv;
    int32_t W, C;
    int32_t io_dtype;
    float qk_scale;
    float l2_eps;
    int32_t gate_dk;     /* 0: g is [L][B][T][Hv]; 1: g is [L][B][T][Hv][Dk], one decay per key
                            channel (GDN investigation §4 tape layout [B, T, Hv, Dk]):
                            S ← S·diag(g_t) + δ_t k_tᵀ with u = S·diag(g_t)·k_t. Every call
                            takes it; trees with fp32 I/O and d = 128 are limited to T <= 16. */
} gdn_dims;

/*
 * gdn_verify — batched multi-token verification through GDN layers, with the innovation tape.
 *
 * Computes (GDN investigation §2.1 "Conv1D state + gated delta state", §2.2 multi-token
 * verification, §4 tape recording; the update is the standard gated delta rule):
 *   x̂ = concat(conv_state rows 0..W-2, qkv rows 0..T-1) per channel
 *   y[t,c] = silu( sum_{j<W} conv_w[c][j] * x̂[t+j, c] )      (tap W-1 is the current token)
 *   q_t, k_t = L2-normalised q and k heads of y;  v_t = v head of y
 *   per value head, from S = S_0:  u = g_t S k_t;  δ_t = β_t (v_t − u);  S ← g_t S + δ_t k_tᵀ;
 *                                  o_t = qk_scale · S q_t
 * Arguments (device):
 *   qkv        [L][B][T][C]        io_dtype   raw projections of the T verify positions
 *   conv_w     [L][C][W]           io_dtype   depthwise conv taps
 *   conv_state [L][B][W-1][C]      io_dtype   last W-1 raw rows before the round (read only)
 *   g, beta    [L][B][T][Hv]       f32        decay gate in (0,1] and write strength; with
 *                                             d->gate_dk, g is [L][B][T][Hv][Dk] (one decay
 *                                             per key channel, S ← S·diag(g_t) + δ_t k_tᵀ)
 *   state      [L][B][Hv][Dv][Dk]  f32        S_0, row-major: element (i,j) of S — row i in
 *                                             Dv, column j in Dk — is at [i][j] (read only)
 *   out        [L][B][T][Hv][Dv]   io_dtype   o_t
 *   tape_delta [L][B][T][Hv][Dv]   f32        δ_t          (written)
 *   tape_k     [L][B][T][Hk][Dk]   f32        normalised k_t (written)
 * The tape's gate and raw-conv parts are the caller's g and qkv themselves: keep them alive and
 * unchanged until gdn_rollback. state, qkv, conv_w and conv_state must be 16-byte aligned (they
 * are read by TMA / bulk copies); every other pointer aligned to its element size. The tape
 * buffers hold gdn_tape_bytes() bytes in total.
 */
GDN_API int gdn_verify(const gdn_dims* d, const void* qkv, const void* conv_w, const void* conv_state,
               const float* g, const float* beta, const float* state, void* out,
               float* tape_delta, float* tape_k, uint32_t* status, void* stream);

/*
 * gdn_verify_tree — gdn_verify over a draft token tree (GDN investigation §2.2 update note and
 * §8 path 3: tree-aware GDN kernels walk the draft tree through the recurrent state).
 *   parent [B][T] int32: parent node of node v, in [-1, v) (-1 = child of the committed context).
 * Node v starts from its parent's state (S_0 for parent -1); its conv window is its own raw row
 * and its W-1 nearest ancestors' rows, continued into conv_state when the path is shorter.
 * Other arguments and layouts as gdn_verify with T = node count; the tape is per node.
 * With d->gate_dk, fp32 I/O and Dk = 128, T is limited to 16 (GDN_ERR_UNSUPPORTED above).
 * A bad parent sets GDN_STATUS_BAD_PARENT; that sequence's out / tape rows are then unspecified
 * (left unwritten, or computed as if the nodes formed one chain).
 */
GDN_API int gdn_verify_tree(const gdn_dims* d, const int32_t* parent, const void* qkv,
                    const void* conv_w, const void* conv_state, const float* g,
                    const float* beta, const float* state, void* out, float* tape_delta,
                    float* tape_k, uint32_t* status, void* stream);

/*
 * gdn_rollback — tape-replay rollback (GDN investigation §4 "Tape-Replay 回滚"): for every layer
 * and sequence with n = n_acc[b] > 0, replay the accepted steps
 *     S ← g_t S + δ_t k_tᵀ,  t = 0..n-1      (with d->gate_dk: S ← S·diag(g_t) + δ_t k_tᵀ),
 * from the untouched snapshot S_0 and store S_n in place; rebuild the conv state as the last W-1
 * rows of (conv_state ++ qkv rows 0..n-1). n = 0 leaves both untouched. Cost O(n), all L layers
 * in one launch; n is read on the device (no host sync).
 *   n_acc [B] int32 device; tape_delta, tape_k, g, qkv as written/passed to gdn_verify;
 *   state and conv_state are updated in place. n outside [0, T] sets GDN_STATUS_BAD_NACC.
 */
GDN_API int gdn_rollback(const gdn_dims* d, const int32_t* n_acc, const float* tape_delta,
                 const float* tape_k, const float* g, const void* qkv, float* state,
                 void* conv_state, uint32_t* status, void* stream);

/*
 * gdn_rollback_path — gdn_rollback along an accepted tree path: the replayed steps are the nodes
 * path[b][0..n-1] (root-most first) of a gdn_verify_tree call, n = n_acc[b] ≤ P.
 *   path [B][P] int32 device (P = path capacity, e.g. the tree depth).
 */
GDN_API int gdn_rollback_path(const gdn_dims* d, const int32_t* path, int32_t P, const int32_t* n_acc,
                      const float* tape_delta, const float* tape_k, const float* g,
                      const void* qkv, float* state, void* conv_state, uint32_t* status,
                      void* stream);

/*
 * gdn_rollback_verify — the previous round's gdn_rollback and this round's gdn_verify in one pass
 * over the recurrent state (GDN investigation §4 tape replay, §2.2 multi-token verification; the
 * fusion is this library's scheduling, the pages run the two steps apart). Same result as
 *     gdn_rollback(d, n_acc_prev, tape_delta_prev, tape_k_prev, g_prev, qkv_prev, state, conv_state)
 *     gdn_verify  (d, qkv, conv_w, conv_state, g, beta, state, out, tape_delta, tape_k)
 * up to floating-point rounding: the committed state is formed in fp32 as gdn_rollback forms it and
 * the verify products are taken from it. With bf16 I/O, Dk = Dv = 128, T ≤ 8 and Hv ∈ {Hk, 2Hk} it
 * is one kernel that reads each state tile once, commits the previous round's accepted steps where
 * n_acc_prev[b] > 0, writes the tile back and verifies the new round from it; other shapes run the
 * two calls. A round loop is then: gdn_rollback_verify (with the previous round's accept result; a
 * first round passes n_acc_prev = 0), spec_accept; after the last round, gdn_rollback.
 * Speed on GB300: it moves about a quarter fewer bytes than the two calls, but the one kernel
 * runs further below the copy bandwidth than either of them (issue contention between its roles),
 * so today the separate gdn_rollback + gdn_verify calls finish sooner (1.65 against 1.89 ms a
 * round at batch 64, N = 8); it stays for callers that want one launch per round.
 * Arguments: the previous round's n_acc_prev [B], tape_delta_prev, tape_k_prev, g_prev, qkv_prev
 * (as gdn_rollback takes them) and this round's verify arguments (as gdn_verify). state and
 * conv_state are updated in place. tape_delta, tape_k and out must not overlap the previous round's
 * tape, qkv or g. state, qkv, qkv_prev, conv_w, conv_state, tape_delta_prev and tape_k_prev must be
 * 16-byte aligned. n outside [0, T] sets GDN_STATUS_BAD_NACC and commits nothing for that sequence.
 */
GDN_API int gdn_rollback_verify(const gdn_dims* d, const int32_t* n_acc_prev,
                        const float* tape_delta_prev, const float* tape_k_prev,
                        const float* g_prev, const void* qkv_prev, const void* qkv,
                        const void* conv_w, void* conv_state, const float* g, const float* beta,
                        float* state, void* out, float* tape_delta, float* tape_k,
                        uint32_t* status, void* stream);

/* Bytes of tape_delta plus tape_k for the shape d (host only, no GPU). 0 on invalid d. */
GDN_API size_t gdn_tape_bytes(const gdn_dims* d);

/*
 * Shapes of one spec_accept call.
 *  B  sequences;  N  drafts per sequence (logits rows per sequence: N + 1, row i judges draft i,
 *  row N is the bonus row);  V  vocabulary;  dtype  GDN_DTYPE_BF16 or GDN_DTYPE_F32 logits;
 *  row_stride, seq_stride  elements between rows / sequences of logits (row_stride ≥ V; a
 *  seq_stride of 0 lets all sequences share one block of rows). Both multiples of 8 for bf16
 *  and of 4 for f32 (16-byte rows).
 */
typedef struct spec_dims {
    int32_t B, N, V, dtype;
    int64_t row_stride, seq_stride;
} spec_dims;

/*
 * spec_accept — acceptance over the verify logits.
 *
 * SPEC_MODE_GREEDY (xserv docs/25 §2 algorithm; colibrì ch.08 §5 greedy path): with
 * am_i = argmax of row i (lowest index among equal maxima), n = the number of leading drafts with
 * drafts[i] == am_i; out = drafts[0..n-1] ++ am_n (the correction, or the bonus when n = N).
 *
 * SPEC_MODE_SAMPLE (colibrì ch.08 §5 Leviathan rejection sampling with point-mass drafts): per
 * row the target law is p = softmax(row / temperature), realised as integer weights
 *   w_v = floor(2^32 · 2^((float(l_v) − float(max)) · c)),  c = fp32(log2(e) / temperature),
 * with the power of two evaluated by a fixed Cody–Waite + degree-7 polynomial so any
 * implementation of this contract draws bit-identical results. Draw r uniform on [0, Z)
 * (Z = Σ w) from Philox4x32-10 with key = seed and counter = (round mod 2^32, b, row, purpose);
 * accept draft i iff r < w[draft_i]. On the first rejection, ban draft i (weight 0), renormalise
 * and sample the emitted token from what is left; if all N are accepted, sample the bonus from
 * row N. temperature ≤ 0 selects greedy.
 *
 * Arguments:
 *   logits     device, laid out by d (row i of sequence b at b*seq_stride + i*row_stride)
 *   drafts     [B][N] int32 device; a token outside [0, V) sets GDN_STATUS_BAD_TOKEN and that
 *              sequence reports n = 0 and out = {-1...}
 *   workspace  device scratch of spec_workspace_bytes(d, mode) bytes, 16-byte aligned; no state
 *              is kept in it between calls
 *   n_acc      [B] int32 device: accepted drafts n in [0, N]
 *   out_tokens [B][N+1] int32 device: the n accepted drafts, then the correction/bonus token,
 *              then -1 padding
 */
GDN_API int spec_accept(const spec_dims* d, const void* logits, const int32_t* drafts, int32_t mode,
                float temperature, uint64_t seed, uint64_t round, void* workspace,
                size_t workspace_bytes, int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                void* stream);

/* Workspace bytes spec_accept needs for d and mode (host only). 0 on invalid d. */
GDN_API size_t spec_workspace_bytes(const spec_dims* d, int32_t mode);

/*
 * spec_stats_accumulate — acceptance statistics for an adaptive speculation switch (colibrì
 * ch.08 §4.1: drafting is turned off once enough drafts were proposed and fewer than one in ten
 * was accepted; the policy itself is the caller's, see speculative_verify_gdn_gb300.adaptive).
 *   B, N    sequences and drafts per sequence of the spec_accept / spec_accept_tree call
 *   n_acc   [B] int32 device, the accepted counts that call wrote (n in [0, N])
 *   stats   [N + 3] uint64 device, accumulated across calls (the caller zeroes it once):
 *           stats[0] += B·N proposed drafts, stats[1] += Σ n accepted drafts,
 *           stats[2 + k] += number of sequences with n = k (k = 0 .. N)
 *   status  optional device word: a count outside [0, N] sets GDN_STATUS_BAD_NACC and adds
 *           nothing but its N proposals
 * One small kernel on `stream`; never synchronises. B = 0 is a no-op.
 */
GDN_API int spec_stats_accumulate(int32_t B, int32_t N, const int32_t* n_acc, uint64_t* stats,
                                  uint32_t* status, void* stream);

/*
 * spec_accept_tree — greedy acceptance of the longest matching root-to-leaf path of a draft
 * tree (GDN investigation §2.2 / §8: DDTree verification). Rows: row 0 judges the children of
 * the committed context, row 1+v judges the children of node v. From the context, repeatedly
 * move to the lowest-numbered child whose token equals the argmax of the current row; stop when
 * none matches or after P steps. The argmax of the last row reached is the bonus token.
 *   d          B, N = T (nodes, at most 4096, else GDN_ERR_UNSUPPORTED; rows per sequence are
 *              T + 1), V, dtype, strides as spec_dims
 *   parent     [B][T] int32, tokens [B][T] int32 device (tree of gdn_verify_tree)
 *   path       [B][P] int32 device: accepted nodes root-most first, -1 padded
 *   n_acc      [B] int32; out_tokens [B][P+1] int32 (path tokens, bonus, -1 padding)
 * workspace as spec_accept with SPEC_MODE_GREEDY.
 */
GDN_API int spec_accept_tree(const spec_dims* d, const void* logits, const int32_t* parent,
                     const int32_t* tokens, int32_t P, void* workspace, size_t workspace_bytes,
                     int32_t* path, int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                     void* stream);

/*
 * spec_accept_static — spec_accept without a caller-provided workspace, for callers that cannot
 * allocate device memory (code that only receives device pointers from its host framework, runs
 * where cudaMalloc is not allowed, or must not allocate on this path). The pages describe no such
 * call; it is a deployment convenience of this library.
 *
 * The scratch is a fixed array of GDN_STATIC_SCRATCH_BYTES bytes in the library's device image,
 * held by every device that loads the library until the process exits; nothing is allocated or
 * freed. Arguments and results are those of spec_accept. Limits:
 *  - a shape whose spec_workspace_bytes() exceeds GDN_STATIC_SCRATCH_BYTES returns
 *    GDN_ERR_UNSUPPORTED (use spec_accept with a workspace instead);
 *  - all calls on a device share the array: calls whose kernels may overlap on the GPU (different
 *    streams without ordering) race and must not be issued;
 *  - the first call on each device looks up the array's device address with that device current,
 *    and looks it up again once the device's context has changed (after cudaDeviceReset); make
 *    the first call on a device, and the first after a reset, outside of any stream capture.
 */
#define GDN_STATIC_SCRATCH_BYTES (1u << 20)
GDN_API int spec_accept_static(const spec_dims* d, const void* logits, const int32_t* drafts,
                               int32_t mode, float temperature, uint64_t seed, uint64_t round,
                               int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                               void* stream);

/* Thread-local message for the last non-OK return on this thread ("" if none). */
GDN_API const char* gdn_last_error(void);

/*
 * gdn_status_check — host-side mapping of a device status word (read back after synchronising the
 * stream the calls ran on) to a return code: GDN_OK for 0, else GDN_ERR_DEVICE_STATUS with the
 * names of the set GDN_STATUS_* bits in gdn_last_error(). Touches no GPU.
 */
GDN_API int gdn_status_check(uint32_t status_word);

/*
 * gdn_set_wait_limit_ns — how long the pipelined verify kernel (bf16, Dk = Dv = 128: gdn_verify,
 * gdn_verify_tree, gdn_rollback_verify) lets one of its on-chip pipeline waits spin before it
 * gives up, sets GDN_STATUS_WAIT_TIMEOUT and lets the CTA run to its end without waiting (the
 * call's outputs are then undefined). 0 restores the default of one second. The waits that drain
 * copies and tensor-core work before a CTA exits always keep the full second. Process-wide, read
 * at each launch; a hook for testing the give-up path (a limit of a few nanoseconds makes it run
 * out). Host only; always GDN_OK. The pages have no counterpart.
 */
GDN_API int gdn_set_wait_limit_ns(uint64_t ns);

/* ---- full-attention layers of the hybrid ------------------------------------------------ */
/*
 * Shapes of one attn_verify call (GDN investigation §2.1: the hybrid's other layer type is
 * standard multi-head attention over a KV cache; §2.2: its N verify positions run in parallel).
 *  L    attention layers covered by the call        B  sequences      T  verify positions
 *  Hq, Hkv  query and kv heads, Hq a multiple of Hkv; query head h reads kv head h / (Hq/Hkv)
 *  D    head dim (built for 128 and 256)            T * (Hq / Hkv) <= 128
 *  ctx  cache capacity in rows per (layer, sequence, kv head), a multiple of 128
 *  scale  multiplies q·k (1/sqrt(D) for the usual scaled dot product)
 */
typedef struct attn_dims {
    int32_t L, B, T;
    int32_t Hq, Hkv, D;
    int32_t ctx;
    float scale;
} attn_dims;

/*
 * attn_verify — the T verify positions of every attention layer in one launch sequence:
 * append their key / value rows to the cache at rows kv_len[b] .. kv_len[b]+T-1, then
 *     o(i, h) = Σ_{j ≤ kv_len[b]+i} softmax_j(scale · q(i, h)·k_j) v_j
 * over kv head h / (Hq/Hkv) (causal inside the new block). kv_len is read on the device and is
 * not changed (attn_truncate moves it once the round is accepted).
 * Arguments (device, bf16 unless noted):
 *   q         [L][B][T][Hq][D]
 *   k_new, v_new [L][B][T][Hkv][D]   the positions' projected keys / values
 *   k_cache   [L][B][Hkv][ctx][D]    token-major: row j is the key of position j
 *   vt_cache  [L][B][Hkv][ctx/128][D][128]  value cache transposed per 128-position tile: the
 *                                    value of position j is column j % 128 of tile j / 128 (both
 *                                    tensor-core operands then read K-major, and every tile is
 *                                    one contiguous block)
 *   kv_len    [B] int32              committed rows per sequence (the same for every layer)
 *   out       [L][B][T][Hq][D]
 *   workspace attn_workspace_bytes(d) bytes (16-byte aligned; NULL when that is 0)
 * Rows of the caches at or beyond kv_len[b] + T are never attended, but their values are
 * multiplied by zero weights: keep them finite (allocate the caches zeroed). q, k_new, v_new,
 * k_cache and vt_cache must be 16-byte aligned (TMA and 16-byte copies); otherwise
 * GDN_ERR_INVALID_ARG. A sequence with kv_len[b] outside [0, ctx − T] sets
 * GDN_STATUS_BAD_LEN and is skipped (cache and out rows unwritten).
 */
GDN_API int attn_verify(const attn_dims* d, const void* q, const void* k_new, const void* v_new,
                        void* k_cache, void* vt_cache, const int32_t* kv_len, void* out,
                        void* workspace, size_t workspace_bytes, uint32_t* status, void* stream);

/* Scratch bytes attn_verify needs for d (partial results when the cache is split across CTAs). */
GDN_API size_t attn_workspace_bytes(const attn_dims* d);

/*
 * attn_truncate — KV truncation on reject: kv_len[b] += n_acc[b] (the accepted drafts' rows stay,
 * the rest are dropped by the length alone and overwritten next round). n_acc, kv_len [B] int32
 * device; n outside [0, T] sets GDN_STATUS_BAD_NACC and leaves kv_len[b].
 */
GDN_API int attn_truncate(int32_t B, int32_t T, const int32_t* n_acc, int32_t* kv_len,
                          uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDNSPEC_H */
