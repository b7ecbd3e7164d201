// api.cu — the extern "C" boundary of libgdnspec: argument validation, shape dispatch and the
// thread-local error message. Every entry point only enqueues work on the caller's stream; none
// allocates, frees or synchronises. See include/gdnspec.h for the contract of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "../../include/gdnspec.h"
#include "kernels.h"
#include "attn.h"

#include <atomic>

namespace {

thread_local char g_err[512] = "";
// gdn_set_wait_limit_ns: give-up time of the pipelined verify kernel's pipeline waits (0: 1 s)
std::atomic<unsigned long long> g_wait_ns{0};

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GDN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t io_size(int dtype) { return dtype == GDN_DTYPE_BF16 ? 2 : 4; }

// Validates a gdn_dims. Returns GDN_OK, or an error code with g_err set.
int check_dims(const gdn_dims* d) {
    if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
    if (d->L < 0 || d->B < 0 || d->T < 0)
        return fail(GDN_ERR_INVALID_ARG, "negative L/B/T (%d, %d, %d)", d->L, d->B, d->T);
    if (d->Hk < 1 || d->Hv < 1 || d->Hv % d->Hk != 0)
        return fail(GDN_ERR_INVALID_ARG, "Hv (%d) must be a positive multiple of Hk (%d)", d->Hv,
                    d->Hk);
    if (d->W < 1 || d->W > 4) return fail(GDN_ERR_UNSUPPORTED, "conv width W=%d not in 1..4", d->W);
    if (d->io_dtype != GDN_DTYPE_BF16 && d->io_dtype != GDN_DTYPE_F32)
        return fail(GDN_ERR_INVALID_ARG, "io_dtype %d unknown", d->io_dtype);
    if (d->Dk != d->Dv || (d->Dk != 32 && d->Dk != 64 && d->Dk != 128))
        return fail(GDN_ERR_UNSUPPORTED, "head dims Dk=%d Dv=%d: built for Dk == Dv in {32,64,128}",
                    d->Dk, d->Dv);
    const long long C = 2LL * d->Hk * d->Dk + 1LL * d->Hv * d->Dv;
    if (d->C != C) return fail(GDN_ERR_INVALID_ARG, "C=%d but 2*Hk*Dk + Hv*Dv = %lld", d->C, C);
    if (d->T > 32) return fail(GDN_ERR_UNSUPPORTED, "T=%d > 32 positions per call", d->T);
    if (d->B > 65535 || d->L > 65535 || d->Hv > 65535)
        return fail(GDN_ERR_UNSUPPORTED, "grid limits: B, L, Hv must be <= 65535");
    if (!(d->l2_eps >= 0.f) || !std::isfinite(d->qk_scale))
        return fail(GDN_ERR_INVALID_ARG, "l2_eps must be >= 0 and qk_scale finite");
    if (d->gate_dk != 0 && d->gate_dk != 1)
        return fail(GDN_ERR_INVALID_ARG, "gate_dk=%d must be 0 or 1", d->gate_dk);
    return GDN_OK;
}

bool empty(const gdn_dims* d) { return d->L == 0 || d->B == 0 || d->T == 0; }

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// 2-D view of the state: rows (l, b, h, i) x columns j; boxes of 32 columns x Dv rows with the
// 128-byte swizzle, which is the tensor cores' K-major operand layout.
int state_tensor_map(const gdn_dims* d, const float* state, CUtensorMap* map) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    const cuuint64_t rows = cuuint64_t(d->L) * d->B * d->Hv * d->Dv;
    cuuint64_t dims[2] = {cuuint64_t(d->Dk), rows};
    cuuint64_t strides[1] = {cuuint64_t(d->Dk) * 4};
    cuuint32_t box[2] = {32, cuuint32_t(d->Dv)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(state), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return GDN_OK;
}

// 2-D views of the bf16 inputs for the pipelined verify: qkv rows (l, b, t) x channels, boxes of
// 128 channels x T rows; conv-state rows (l, b, w) x channels, boxes of 128 channels x (W-1) rows.
// Returns false (no error) when the shape does not suit them.
bool input_tensor_maps(const gdn_dims* d, const void* qkv, const void* conv_state,
                       gdn::VerifyMaps* m) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc || d->io_dtype != GDN_DTYPE_BF16 || d->Dk != 128 || d->Dv != 128 || d->T > 256 ||
        (size_t(d->C) * 2) % 16 != 0)
        return false;
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t strides[1] = {cuuint64_t(d->C) * 2};
    cuuint64_t qdims[2] = {cuuint64_t(d->C), cuuint64_t(d->L) * d->B * d->T};
    cuuint32_t qbox[2] = {128, cuuint32_t(d->T)};
    if (enc(&m->qkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), qdims, strides, qbox,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (d->W > 1) {
        cuuint64_t cdims[2] = {cuuint64_t(d->C), cuuint64_t(d->L) * d->B * (d->W - 1)};
        cuuint32_t cbox[2] = {128, cuuint32_t(d->W - 1)};
        if (enc(&m->conv_state, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(conv_state),
                cdims, strides, cbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    } else {
        m->conv_state = m->qkv;   // never read: no conv-state rows when W == 1
    }
    return true;
}

int verify_common(const gdn_dims* d, const int32_t* parent, const void* qkv, const void* conv_w,
                  const void* conv_state, const float* g, const float* beta, const float* state,
                  void* out, float* tape_delta, float* tape_k, uint32_t* status, void* stream,
                  bool tree) {
    int rc = check_dims(d);
    if (rc) return rc;
    if (tree && d->gate_dk && d->io_dtype == GDN_DTYPE_F32 && d->Dk == 128 && d->T > 16)
        return fail(GDN_ERR_UNSUPPORTED,
                    "gdn_verify_tree with per-key-channel gates, fp32 I/O and d=128: T <= 16");
    if (empty(d)) return GDN_OK;
    if (!qkv || !conv_w || !g || !beta || !state || !out || !tape_delta || !tape_k ||
        (d->W > 1 && !conv_state) || (tree && !parent))
        return fail(GDN_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(state, 16) || !aligned(qkv, 16) || !aligned(conv_w, 16) ||
        (conv_state && !aligned(conv_state, 16)))
        return fail(GDN_ERR_INVALID_ARG,
                    "state, qkv, conv_w and conv_state must be 16-byte aligned (TMA / bulk copies)");
    const size_t es = io_size(d->io_dtype);
    if (!aligned(out, es) || !aligned(g, 4) || !aligned(beta, 4) || !aligned(tape_delta, 4) ||
        !aligned(tape_k, 4))
        return fail(GDN_ERR_INVALID_ARG, "misaligned tensor pointer");
    gdn::VerifyArgs a{};
    a.L = d->L; a.B = d->B; a.T = d->T; a.Hk = d->Hk; a.Hv = d->Hv; a.W = d->W; a.C = d->C;
    a.qk_scale = d->qk_scale; a.l2_eps = d->l2_eps;
    a.qkv = qkv; a.conv_w = conv_w; a.conv_state = conv_state; a.g = g; a.beta = beta;
    a.state = state; a.out = out; a.tape_delta = tape_delta; a.tape_k = tape_k;
    a.parent = tree ? parent : nullptr; a.status = status; a.gate_dk = d->gate_dk;
    a.wait_ns = g_wait_ns.load();
    gdn::VerifyMaps maps;
    rc = state_tensor_map(d, state, &maps.state);
    if (rc) return rc;
    maps.inputs_ok = input_tensor_maps(d, qkv, conv_state, &maps);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = d->io_dtype == GDN_DTYPE_BF16
                        ? gdn::launch_verify_bf16(a, maps, d->Dk, tree, s)
                        : gdn::launch_verify_f32(a, maps, d->Dk, tree, s);
    if (e != cudaSuccess) return cuda_fail(e, tree ? "gdn_verify_tree launch" : "gdn_verify launch");
    return GDN_OK;
}

// 2-D view of the previous round's qkv for the fused rollback + verify: rows (l, b, t) x channels,
// boxes of 128 channels x (W-1) rows (the last W-1 raw rows of the new conv window).
bool prev_qkv_map(const gdn_dims* d, const void* qkv_prev, gdn::VerifyMaps* m) {
    if (d->W == 1) {
        m->qkv_prev = m->qkv;      // never read
        return true;
    }
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t strides[1] = {cuuint64_t(d->C) * 2};
    cuuint64_t dims[2] = {cuuint64_t(d->C), cuuint64_t(d->L) * d->B * d->T};
    cuuint32_t box[2] = {128, cuuint32_t(d->W - 1)};
    return enc(&m->qkv_prev, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv_prev), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void* p, size_t n, const void* q, size_t m) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return n && m && a < b + m && b < a + n;
}

int rollback_common(const gdn_dims* d, const int32_t* path, int32_t P, const int32_t* n_acc,
                    const float* tape_delta, const float* tape_k, const float* g, const void* qkv,
                    float* state, void* conv_state, uint32_t* status, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if (path && P < 0) return fail(GDN_ERR_INVALID_ARG, "path capacity P=%d < 0", P);
    if (empty(d) || (path && P == 0)) return GDN_OK;
    if (!n_acc || !tape_delta || !tape_k || !g || !qkv || !state || (d->W > 1 && !conv_state))
        return fail(GDN_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(state, 16) || !aligned(tape_delta, 16))
        return fail(GDN_ERR_INVALID_ARG, "state and tape_delta must be 16-byte aligned");
    const size_t es = io_size(d->io_dtype);
    if (!aligned(qkv, es) || (conv_state && !aligned(conv_state, es)) || !aligned(tape_k, 4) ||
        !aligned(g, 4) || !aligned(n_acc, 4) || (path && !aligned(path, 4)))
        return fail(GDN_ERR_INVALID_ARG, "misaligned tensor pointer");
    gdn::RollbackArgs a{};
    a.L = d->L; a.B = d->B; a.T = d->T; a.Hk = d->Hk; a.Hv = d->Hv; a.W = d->W; a.C = d->C;
    a.P = path ? P : 0;
    a.n_acc = n_acc; a.path = path; a.tape_delta = tape_delta; a.tape_k = tape_k; a.g = g;
    a.qkv = qkv; a.state = state; a.conv_state = conv_state; a.status = status;
    a.gate_dk = d->gate_dk;
    cudaError_t e = gdn::launch_rollback(a, d->Dk, d->io_dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, path ? "gdn_rollback_path launch" : "gdn_rollback launch");
    return GDN_OK;
}

int check_spec(const spec_dims* d) {
    if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
    if (d->B < 0 || d->N < 0 || d->V < 1)
        return fail(GDN_ERR_INVALID_ARG, "bad B=%d N=%d V=%d", d->B, d->N, d->V);
    if (d->dtype != GDN_DTYPE_BF16 && d->dtype != GDN_DTYPE_F32)
        return fail(GDN_ERR_INVALID_ARG, "logits dtype %d unknown", d->dtype);
    const int64_t vecn = d->dtype == GDN_DTYPE_BF16 ? 8 : 4;
    if (d->row_stride < d->V || d->row_stride % vecn != 0)
        return fail(GDN_ERR_INVALID_ARG, "row_stride %lld must be >= V and a multiple of %lld",
                    (long long)d->row_stride, (long long)vecn);
    if (d->seq_stride < 0 || d->seq_stride % vecn != 0)
        return fail(GDN_ERR_INVALID_ARG, "seq_stride %lld must be >= 0 and a multiple of %lld",
                    (long long)d->seq_stride, (long long)vecn);
    if (1LL * d->B * (d->N + 1) > 0x7fffffffLL)
        return fail(GDN_ERR_UNSUPPORTED, "B*(N+1) rows exceed the grid");
    return GDN_OK;
}

// tiles of one warp's 16-byte loads: 32 vectors of 8 bf16 or 4 fp32 logits
int tile_elems(int dtype) { return dtype == GDN_DTYPE_BF16 ? 256 : 128; }

size_t ws_bytes(const spec_dims* d, int32_t mode) {
    const int rows = d->B * (d->N + 1);
    int CH, CS;
    gdn::accept_chunking(rows, d->V, &CH, &CS);
    const size_t keys = size_t(rows) * CH * 8;
    if (mode == SPEC_MODE_SAMPLE) {
        const int TE = tile_elems(d->dtype), NT = (CS + TE - 1) / TE;
        return keys * 2 + size_t(rows) * 8 + keys * NT;
    }
    return keys;
}

gdn::AcceptArgs accept_args(const spec_dims* d, const void* logits, void* workspace) {
    gdn::AcceptArgs a{};
    a.B = d->B; a.N = d->N; a.V = d->V;
    const int rows = d->B * (d->N + 1);
    gdn::accept_chunking(rows, d->V, &a.CH, &a.CS);
    a.row_stride = d->row_stride; a.seq_stride = d->seq_stride;
    a.logits = logits;
    auto* ws = static_cast<unsigned long long*>(workspace);
    a.ws_key = ws;
    a.ws_sum = ws + size_t(rows) * a.CH;
    a.ws_wd = ws + size_t(rows) * a.CH * 2;
    const int TE = tile_elems(d->dtype);
    a.NT = (a.CS + TE - 1) / TE;
    a.ws_tile = a.ws_wd + rows;      // used by the sampling mode only (sized by ws_bytes)
    return a;
}

int check_attn(const attn_dims* d) {
    if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
    if (d->L < 0 || d->B < 0 || d->T < 0)
        return fail(GDN_ERR_INVALID_ARG, "negative L/B/T (%d, %d, %d)", d->L, d->B, d->T);
    if (d->Hkv < 1 || d->Hq < 1 || d->Hq % d->Hkv != 0)
        return fail(GDN_ERR_INVALID_ARG, "Hq (%d) must be a positive multiple of Hkv (%d)", d->Hq,
                    d->Hkv);
    if (d->D != 128 && d->D != 256)
        return fail(GDN_ERR_UNSUPPORTED, "attention head dim D=%d: built for 128 and 256", d->D);
    if (1LL * d->T * (d->Hq / d->Hkv) > 128)
        return fail(GDN_ERR_UNSUPPORTED, "T * Hq/Hkv = %lld query rows per kv head > 128",
                    1LL * d->T * (d->Hq / d->Hkv));
    if (d->ctx < 128 || d->ctx % 128 != 0)
        return fail(GDN_ERR_UNSUPPORTED, "cache capacity ctx=%d: needs a positive multiple of 128",
                    d->ctx);
    if (d->T > d->ctx) return fail(GDN_ERR_INVALID_ARG, "T=%d > ctx=%d", d->T, d->ctx);
    if (!std::isfinite(d->scale)) return fail(GDN_ERR_INVALID_ARG, "scale must be finite");
    const long long heads = 1LL * d->L * d->B * d->Hkv;
    if (heads * d->ctx >= (1LL << 31) || heads * (d->ctx / 128) * d->D >= (1LL << 31) || d->B > 65535 ||
        d->L > 65535)
        return fail(GDN_ERR_UNSUPPORTED, "attention caches too large for 32-bit row indices");
    return GDN_OK;
}

// Work plan of the attention kernels, whose CTAs each take one SM: whole waves of units over the
// 152 SMs of a GB300 run whole (one CTA per unit); the units left over are split into key ranges
// so that the last wave is filled with short CTAs (at most one wave of them), and only those
// units' partial results go through the workspace and the combine kernel. The plan depends on
// the shapes alone, so the workspace size does too.
void attn_plan(const attn_dims* d, int* n_full, int* splits, int* tiles_per_split) {
    constexpr long long kSMs = 152;
    const long long units = 1LL * d->L * d->B * d->Hkv;
    const int cap = (d->ctx + 127) / 128;
    const long long rest = units % kSMs;
    *n_full = int(units - rest);
    *splits = 1;
    *tiles_per_split = cap;
    if (rest == 0 || cap <= 1) {
        *n_full = int(units);
        return;
    }
    long long sp = kSMs / rest;
    if (sp > cap) sp = cap;
    if (sp < 1) sp = 1;
    const int t = int((cap + sp - 1) / sp);
    *tiles_per_split = t;
    *splits = (cap + t - 1) / t;
    if (*splits == 1) *n_full = int(units);
}

size_t attn_ws_bytes(const attn_dims* d) {
    int nf, sp, tps;
    attn_plan(d, &nf, &sp, &tps);
    const long long tail = 1LL * d->L * d->B * d->Hkv - nf;
    if (sp <= 1 || tail <= 0) return 0;
    const size_t rows = size_t(sp) * size_t(tail) * size_t(d->T) * (d->Hq / d->Hkv);
    return rows * (size_t(d->D) + 2) * 4;
}

}  // namespace

namespace gdn {
int report_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}
}  // namespace gdn

extern "C" {

int gdn_verify(const gdn_dims* d, const void* qkv, const void* conv_w, const void* conv_state,
               const float* g, const float* beta, const float* state, void* out,
               float* tape_delta, float* tape_k, uint32_t* status, void* stream) {
    return verify_common(d, nullptr, qkv, conv_w, conv_state, g, beta, state, out, tape_delta,
                         tape_k, status, stream, false);
}

int gdn_verify_tree(const gdn_dims* d, const int32_t* parent, const void* qkv,
                    const void* conv_w, const void* conv_state, const float* g,
                    const float* beta, const float* state, void* out, float* tape_delta,
                    float* tape_k, uint32_t* status, void* stream) {
    return verify_common(d, parent, qkv, conv_w, conv_state, g, beta, state, out, tape_delta,
                         tape_k, status, stream, true);
}

int gdn_rollback(const gdn_dims* d, const int32_t* n_acc, const float* tape_delta,
                 const float* tape_k, const float* g, const void* qkv, float* state,
                 void* conv_state, uint32_t* status, void* stream) {
    return rollback_common(d, nullptr, 0, n_acc, tape_delta, tape_k, g, qkv, state, conv_state,
                           status, stream);
}

int gdn_rollback_path(const gdn_dims* d, const int32_t* path, int32_t P, const int32_t* n_acc,
                      const float* tape_delta, const float* tape_k, const float* g,
                      const void* qkv, float* state, void* conv_state, uint32_t* status,
                      void* stream) {
    if (!path) return fail(GDN_ERR_INVALID_ARG, "path is NULL");
    return rollback_common(d, path, P, n_acc, tape_delta, tape_k, g, qkv, state, conv_state,
                           status, stream);
}

size_t gdn_tape_bytes(const gdn_dims* d) {
    if (check_dims(d) != GDN_OK) return 0;
    const size_t lbt = size_t(d->L) * d->B * d->T;
    return lbt * (size_t(d->Hv) * d->Dv + size_t(d->Hk) * d->Dk) * 4;
}

int spec_accept(const spec_dims* d, const void* logits, const int32_t* drafts, int32_t mode,
                float temperature, uint64_t seed, uint64_t round, void* workspace,
                size_t workspace_bytes, int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                void* stream) {
    int rc = check_spec(d);
    if (rc) return rc;
    if (mode != SPEC_MODE_GREEDY && mode != SPEC_MODE_SAMPLE)
        return fail(GDN_ERR_INVALID_ARG, "mode %d unknown", mode);
    if (mode == SPEC_MODE_SAMPLE && !(temperature > 0.f)) mode = SPEC_MODE_GREEDY;
    if (mode == SPEC_MODE_SAMPLE && !std::isfinite(temperature))
        return fail(GDN_ERR_INVALID_ARG, "temperature must be finite");
    if (d->B == 0) return GDN_OK;
    if (!logits || !n_acc || !out_tokens || !workspace || (d->N > 0 && !drafts))
        return fail(GDN_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(logits, 16) || !aligned(workspace, 16))
        return fail(GDN_ERR_INVALID_ARG, "logits and workspace must be 16-byte aligned");
    const size_t need = ws_bytes(d, mode);
    if (workspace_bytes < need)
        return fail(GDN_ERR_INVALID_ARG, "workspace %zu bytes < %zu required", workspace_bytes, need);
    gdn::AcceptArgs a = accept_args(d, logits, workspace);
    a.drafts = drafts; a.n_acc = n_acc; a.out_tokens = out_tokens; a.status = status;
    a.seed = seed; a.round = uint32_t(round);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (mode == SPEC_MODE_SAMPLE) {
        a.c = float((1.0 / std::log(2.0)) / double(temperature));
        e = gdn::launch_accept_sample(a, d->dtype, s);
    } else {
        e = gdn::launch_accept_greedy(a, d->dtype, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "spec_accept launch");
    return GDN_OK;
}

int spec_stats_accumulate(int32_t B, int32_t N, const int32_t* n_acc, uint64_t* stats,
                          uint32_t* status, void* stream) {
    if (B < 0 || N < 0) return fail(GDN_ERR_INVALID_ARG, "B = %d, N = %d", B, N);
    if (N > 64) return fail(GDN_ERR_UNSUPPORTED, "N = %d > 64", N);
    if (B == 0) return GDN_OK;
    if (!n_acc || !stats) return fail(GDN_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(n_acc, 4) || !aligned(stats, 8))
        return fail(GDN_ERR_INVALID_ARG, "misaligned n_acc or stats");
    const cudaError_t e =
        gdn::launch_spec_stats(B, N, n_acc, stats, status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "spec_stats_accumulate launch");
    return GDN_OK;
}

size_t spec_workspace_bytes(const spec_dims* d, int32_t mode) {
    if (check_spec(d) != GDN_OK) return 0;
    if (mode != SPEC_MODE_GREEDY && mode != SPEC_MODE_SAMPLE) return 0;
    return ws_bytes(d, mode);
}

int spec_accept_tree(const spec_dims* d, const void* logits, const int32_t* parent,
                     const int32_t* tokens, int32_t P, void* workspace, size_t workspace_bytes,
                     int32_t* path, int32_t* n_acc, int32_t* out_tokens, uint32_t* status,
                     void* stream) {
    int rc = check_spec(d);
    if (rc) return rc;
    if (P < 0) return fail(GDN_ERR_INVALID_ARG, "path capacity P=%d < 0", P);
    if (d->N > 4096) return fail(GDN_ERR_UNSUPPORTED, "tree of %d nodes > 4096", d->N);
    if (d->B == 0) return GDN_OK;
    if (!logits || !n_acc || !out_tokens || !workspace || !path ||
        (d->N > 0 && (!parent || !tokens)))
        return fail(GDN_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(logits, 16) || !aligned(workspace, 16))
        return fail(GDN_ERR_INVALID_ARG, "logits and workspace must be 16-byte aligned");
    const size_t need = ws_bytes(d, SPEC_MODE_GREEDY);
    if (workspace_bytes < need)
        return fail(GDN_ERR_INVALID_ARG, "workspace %zu bytes < %zu required", workspace_bytes, need);
    gdn::AcceptArgs a = accept_args(d, logits, workspace);
    a.drafts = tokens; a.parent = parent; a.P = P;
    a.n_acc = n_acc; a.out_tokens = out_tokens; a.path = path; a.status = status;
    cudaError_t e = gdn::launch_accept_tree(a, d->dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "spec_accept_tree launch");
    return GDN_OK;
}

const char* gdn_last_error(void) { return g_err; }

int gdn_set_wait_limit_ns(uint64_t ns) {
    g_wait_ns.store(ns);
    return GDN_OK;
}

int gdn_status_check(uint32_t status_word) {
    if (status_word == 0) return GDN_OK;
    static const struct {
        uint32_t bit;
        const char* name;
    } kBits[] = {{GDN_STATUS_BAD_NACC, "BAD_NACC (accepted count outside [0, T])"},
                 {GDN_STATUS_BAD_PARENT, "BAD_PARENT (tree parent not in [-1, v))"},
                 {GDN_STATUS_BAD_TOKEN, "BAD_TOKEN (draft / tree token outside [0, V))"},
                 {GDN_STATUS_BAD_PATH, "BAD_PATH (path node out of range)"},
                 {GDN_STATUS_EMPTY_DIST, "EMPTY_DIST (a sampling row with zero total weight)"},
                 {GDN_STATUS_WAIT_TIMEOUT, "WAIT_TIMEOUT (a bounded wait gave up; discard the outputs)"},
                 {GDN_STATUS_BAD_LEN, "BAD_LEN (kv_len outside [0, ctx - T])"}};
    char msg[480];
    int n = snprintf(msg, sizeof msg, "device status 0x%x:", status_word);
    uint32_t known = 0;
    for (const auto& b : kBits) {
        known |= b.bit;
        if ((status_word & b.bit) && n > 0 && size_t(n) < sizeof msg)
            n += snprintf(msg + n, sizeof msg - size_t(n), " %s", b.name);
    }
    if ((status_word & ~known) && n > 0 && size_t(n) < sizeof msg)
        snprintf(msg + n, sizeof msg - size_t(n), " unknown bits 0x%x", status_word & ~known);
    return fail(GDN_ERR_DEVICE_STATUS, "%s", msg);
}

int gdn_rollback_verify(const gdn_dims* d, const int32_t* n_acc_prev, const float* tape_delta_prev,
                        const float* tape_k_prev, const float* g_prev, const void* qkv_prev,
                        const void* qkv, const void* conv_w, void* conv_state, const float* g,
                        const float* beta, float* state, void* out, float* tape_delta,
                        float* tape_k, uint32_t* status, void* stream) {
    int rc = check_dims(d);
    if (rc) return rc;
    if (empty(d)) return GDN_OK;
    // every check of both calls comes first: on an error nothing is enqueued
    if (!n_acc_prev || !tape_delta_prev || !tape_k_prev || !g_prev || !qkv_prev || !qkv || !conv_w ||
        !g || !beta || !state || !out || !tape_delta || !tape_k || (d->W > 1 && !conv_state))
        return fail(GDN_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(state, 16) || !aligned(qkv, 16) || !aligned(conv_w, 16) || !aligned(qkv_prev, 16) ||
        !aligned(tape_delta_prev, 16) || !aligned(tape_k_prev, 16) ||
        (conv_state && !aligned(conv_state, 16)))
        return fail(GDN_ERR_INVALID_ARG,
                    "state, qkv, qkv_prev, conv_w, conv_state and the previous tape must be 16-byte "
                    "aligned (TMA / bulk copies)");
    const size_t es = io_size(d->io_dtype);
    if (!aligned(out, es) || !aligned(g, 4) || !aligned(beta, 4) || !aligned(g_prev, 4) ||
        !aligned(tape_delta, 4) || !aligned(tape_k, 4) || !aligned(n_acc_prev, 4))
        return fail(GDN_ERR_INVALID_ARG, "misaligned tensor pointer");
    const size_t lbt = size_t(d->L) * d->B * d->T;
    const size_t dl_bytes = lbt * d->Hv * d->Dv * 4, k_bytes = lbt * d->Hk * d->Dk * 4;
    const size_t q_bytes = lbt * d->C * es, o_bytes = lbt * d->Hv * d->Dv * es;
    const void* outs[3] = {tape_delta, tape_k, out};
    const size_t out_n[3] = {dl_bytes, k_bytes, o_bytes};
    const void* ins[4] = {tape_delta_prev, tape_k_prev, qkv_prev, g_prev};
    const size_t in_n[4] = {dl_bytes, k_bytes, q_bytes, lbt * d->Hv * (d->gate_dk ? d->Dk : 1) * 4};
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 4; ++j)
            if (overlaps(outs[i], out_n[i], ins[j], in_n[j]))
                return fail(GDN_ERR_INVALID_ARG,
                            "this round's tape / out overlap the previous round's tape, qkv or g");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d->io_dtype == GDN_DTYPE_BF16 && !d->gate_dk) {
        gdn::VerifyArgs a{};
        a.L = d->L; a.B = d->B; a.T = d->T; a.Hk = d->Hk; a.Hv = d->Hv; a.W = d->W; a.C = d->C;
        a.qk_scale = d->qk_scale; a.l2_eps = d->l2_eps;
        a.qkv = qkv; a.conv_w = conv_w; a.conv_state = conv_state; a.g = g; a.beta = beta;
        a.state = state; a.out = out; a.tape_delta = tape_delta; a.tape_k = tape_k;
        a.parent = nullptr; a.status = status;
        a.n_acc_prev = n_acc_prev; a.tape_delta_prev = tape_delta_prev; a.tape_k_prev = tape_k_prev;
        a.g_prev = g_prev; a.qkv_prev = qkv_prev; a.conv_state_out = conv_state;
        a.wait_ns = g_wait_ns.load();
        gdn::VerifyMaps maps;
        rc = state_tensor_map(d, state, &maps.state);
        if (rc) return rc;
        maps.inputs_ok = input_tensor_maps(d, qkv, conv_state, &maps) && prev_qkv_map(d, qkv_prev, &maps);
        cudaError_t e = gdn::launch_rollback_verify_bf16(a, maps, d->Dk, s);
        if (e == cudaSuccess) return GDN_OK;
        if (e != cudaErrorNotSupported) return cuda_fail(e, "gdn_rollback_verify launch");
    }
    // other shapes: the two calls in sequence (same result)
    rc = rollback_common(d, nullptr, 0, n_acc_prev, tape_delta_prev, tape_k_prev, g_prev, qkv_prev,
                         state, conv_state, status, stream);
    if (rc) return rc;
    return verify_common(d, nullptr, qkv, conv_w, conv_state, g, beta, state, out, tape_delta,
                         tape_k, status, stream, false);
}

size_t attn_workspace_bytes(const attn_dims* d) {
    if (check_attn(d) != GDN_OK) return 0;
    return attn_ws_bytes(d);
}

int attn_verify(const attn_dims* d, const void* q, const void* k_new, const void* v_new,
                void* k_cache, void* vt_cache, const int32_t* kv_len, void* out, void* workspace,
                size_t workspace_bytes, uint32_t* status, void* stream) {
    int rc = check_attn(d);
    if (rc) return rc;
    if (d->L == 0 || d->B == 0 || d->T == 0) return GDN_OK;
    if (!q || !k_new || !v_new || !k_cache || !vt_cache || !kv_len || !out)
        return fail(GDN_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(vt_cache, 16))
        return fail(GDN_ERR_INVALID_ARG,
                    "q, k_new, v_new, k_cache and vt_cache must be 16-byte aligned (TMA / vector copies)");
    if (!aligned(out, 2) || !aligned(kv_len, 4))
        return fail(GDN_ERR_INVALID_ARG, "misaligned tensor pointer");
    const size_t need = attn_ws_bytes(d);
    if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return fail(GDN_ERR_INVALID_ARG, "workspace %zu bytes (16-byte aligned) < %zu required",
                    workspace_bytes, need);
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    const cuuint64_t heads = cuuint64_t(d->L) * d->B * d->Hkv;
    cuuint32_t estr[2] = {1, 1};
    cuuint32_t box[2] = {64, 128};
    CUtensorMap kmap, vmap;
    {
        cuuint64_t dims[2] = {cuuint64_t(d->D), heads * cuuint64_t(d->ctx)};
        cuuint64_t strides[1] = {cuuint64_t(d->D) * 2};
        if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k_cache, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K cache");
    }
    {
        cuuint64_t dims[2] = {128, heads * cuuint64_t(d->ctx / 128) * cuuint64_t(d->D)};
        cuuint64_t strides[1] = {256};
        if (enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vt_cache, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled failed for the V cache");
    }
    gdn::AttnArgs a{};
    a.L = d->L; a.B = d->B; a.T = d->T; a.Hq = d->Hq; a.Hkv = d->Hkv; a.D = d->D; a.ctx = d->ctx;
    a.group = d->Hq / d->Hkv;
    a.nq = d->T * a.group;
    a.units = d->L * d->B * d->Hkv;
    attn_plan(d, &a.n_full, &a.splits, &a.tiles_per_split);
    a.sl2 = float(double(d->scale) * 1.4426950408889634);
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k_new = static_cast<const __nv_bfloat16*>(k_new);
    a.v_new = static_cast<const __nv_bfloat16*>(v_new);
    a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
    a.vt_cache = static_cast<__nv_bfloat16*>(vt_cache);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.kv_len = kv_len;
    a.status = status;
    if (a.splits > 1 && a.units > a.n_full) {
        a.ws_o = static_cast<float*>(workspace);
        a.ws_ml = a.ws_o + size_t(a.splits) * size_t(a.units - a.n_full) * a.nq * d->D;
    }
    if (1LL * a.n_full + 1LL * (a.units - a.n_full) * a.splits >= (1LL << 31))
        return fail(GDN_ERR_UNSUPPORTED, "attention grid too large");
    const cudaError_t e = gdn::launch_attn_verify(a, kmap, vmap, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_verify launch");
    return GDN_OK;
}

int attn_truncate(int32_t B, int32_t T, const int32_t* n_acc, int32_t* kv_len, uint32_t* status,
                  void* stream) {
    if (B < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "B = %d, T = %d", B, T);
    if (B == 0) return GDN_OK;
    if (!n_acc || !kv_len) return fail(GDN_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(n_acc, 4) || !aligned(kv_len, 4))
        return fail(GDN_ERR_INVALID_ARG, "misaligned n_acc or kv_len");
    const cudaError_t e =
        gdn::launch_attn_truncate(B, T, n_acc, kv_len, status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attn_truncate launch");
    return GDN_OK;
}

}  // extern "C"
