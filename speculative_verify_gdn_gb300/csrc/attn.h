// attn.h — launch interface of the attention-layer kernels (attn.cu), kept apart from the GDN
// kernels' header so that each side's sources change independently.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Attention-layer verify (attn.cu). nq = T·group query rows per kv head; units = L·B·Hkv; the
// keys of a unit are cut into `splits` ranges of `tiles_per_split` 128-key tiles; ws_o / ws_ml
// hold the per-split partials when splits > 1. sl2 = scale·log2(e).
struct AttnArgs {
    int L, B, T, Hq, Hkv, D, ctx, group, nq, units, splits, tiles_per_split;
    int n_full;                       // units 0 .. n_full-1 run whole (one CTA each); the others
                                      // are split into `splits` key ranges of tiles_per_split
    float sl2;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_new;
    const __nv_bfloat16* v_new;
    __nv_bfloat16* k_cache;
    __nv_bfloat16* vt_cache;
    __nv_bfloat16* out;
    const int32_t* kv_len;
    float* ws_o;
    float* ws_ml;
    uint32_t* status;
};
// kmap: the K cache as rows [L·B·Hkv·ctx] x D; vmap: the tile-transposed V cache as rows
// [L·B·Hkv·(ctx/128)·D] x 128; both bf16, boxes 64 x 128, 128-byte swizzle.
cudaError_t launch_attn_verify(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               cudaStream_t s);
cudaError_t launch_attn_truncate(int B, int T, const int32_t* n_acc, int32_t* kv_len,
                                 uint32_t* status, cudaStream_t s);

}  // namespace gdn
