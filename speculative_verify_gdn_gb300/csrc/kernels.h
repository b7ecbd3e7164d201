// kernels.h — host-side launch entry points of the gdnspec kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

struct VerifyArgs {
    int L, B, T, Hk, Hv, W, C;
    float qk_scale, l2_eps;
    const void* qkv;
    const void* conv_w;
    const void* conv_state;
    const float* g;
    const float* beta;
    const float* state;
    void* out;
    float* tape_delta;
    float* tape_k;
    const int32_t* parent;   // tree only (null for the chain)
    uint32_t* status;
    int gate_dk;             // g is [L][B][T][Hv][Dk] (per key channel) instead of [..][Hv]
    // gdn_rollback_verify only (null otherwise): the previous round's accepted counts [B], tape
    // (δ [L][B][T][Hv][Dv], k [L][B][T][Hk][Dk]), gates [L][B][T][Hv] and raw rows [L][B][T][C];
    // the state and conv_state buffers are then updated in place
    const int32_t* n_acc_prev;
    const float* tape_delta_prev;
    const float* tape_k_prev;
    const float* g_prev;
    const void* qkv_prev;
    void* conv_state_out;
    uint64_t wait_ns;         // give-up time of the pipelined kernel's pipeline waits (0: 1 s)
};

// TMA maps of one verify call. `state`: rows [L*B*Hv*Dv] x cols [Dk], 32 x Dv boxes, 128-byte
// swizzle. `qkv`: rows [L*B*T] x channels [C], boxes of 128 channels x T rows; `conv_state`: rows
// [L*B*(W-1)] x channels [C], boxes of 128 channels x (W-1) rows (no swizzle). `inputs_ok` is false
// when the two input maps could not be made (then only kernels that do not use them run).
struct VerifyMaps {
    CUtensorMap state;
    CUtensorMap qkv;
    CUtensorMap conv_state;
    CUtensorMap qkv_prev;    // gdn_rollback_verify: previous round's qkv, boxes of 128 x (W-1)
    bool inputs_ok;
};

// verify: D = Dk = Dv. One translation unit per element type of qkv / conv / out.
cudaError_t launch_verify_bf16(const VerifyArgs& a, const VerifyMaps& m, int D, bool tree,
                               cudaStream_t s);
cudaError_t launch_verify_f32(const VerifyArgs& a, const VerifyMaps& m, int D, bool tree,
                              cudaStream_t s);
// gdn_rollback_verify in one kernel when the shape suits the pipelined kernel (bf16, D = 128,
// T <= 8, Hv in {Hk, 2Hk}); returns cudaErrorNotSupported otherwise (the caller then runs the
// rollback and the verify as two launches).
cudaError_t launch_rollback_verify_bf16(const VerifyArgs& a, const VerifyMaps& m, int D,
                                        cudaStream_t s);

struct RollbackArgs {
    int L, B, T, Hk, Hv, W, C, P;
    const int32_t* n_acc;
    const int32_t* path;      // null for the chain
    const float* tape_delta;
    const float* tape_k;
    const float* g;
    const void* qkv;
    float* state;
    void* conv_state;
    uint32_t* status;
    int gate_dk;              // g per key channel [L][B][T][Hv][Dk]
};
cudaError_t launch_rollback(const RollbackArgs& a, int D, int io_dtype, cudaStream_t s);

struct AcceptArgs {
    int B, N, V;              // N = drafts (chain) or nodes (tree); rows per sequence = N + 1
    int CH, CS;               // vocabulary chunks per row and chunk length
    int64_t row_stride, seq_stride;
    const void* logits;
    const int32_t* drafts;    // chain drafts, or the tree's node tokens
    const int32_t* parent;    // tree only
    int P;                    // tree path capacity
    float c;                  // sampling: fp32(log2(e) / temperature)
    uint64_t seed;
    uint32_t round;
    unsigned long long* ws_key;
    unsigned long long* ws_sum;
    unsigned long long* ws_wd;
    unsigned long long* ws_tile;   // sampling: weight sums of 32-vector tiles [rows][CH][NT]
    int NT;                        // tiles per chunk
    int32_t* n_acc;
    int32_t* out_tokens;
    int32_t* path;
    uint32_t* status;
};

// Opts `kernel` in to `bytes` of dynamic shared memory in the current context (remembered per
// context and kernel under a mutex, so a second GPU or a reset device is set up again).
cudaError_t smem_optin(const void* kernel, size_t bytes);
// SM count of the current device (looked up once per device).
cudaError_t device_sm_count(int* n);
// Unique id (+1) of the calling thread's current CUDA context; 0 if none is current or the
// driver does not expose it.
unsigned long long current_context_id();

// Sets the calling thread's gdn_last_error() message and returns `code`.
int report_error(int code, const char* fmt, ...);

// Vocabulary chunking shared by spec_accept's workspace size query and its launches.
void accept_chunking(int rows, int V, int* CH, int* CS);

cudaError_t launch_accept_greedy(const AcceptArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_accept_sample(const AcceptArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_accept_tree(const AcceptArgs& a, int dtype, cudaStream_t s);
// acceptance counters (spec_stats_accumulate); N <= 64
cudaError_t launch_spec_stats(int B, int N, const int32_t* n_acc, uint64_t* stats, uint32_t* status,
                              cudaStream_t s);

}  // namespace gdn
