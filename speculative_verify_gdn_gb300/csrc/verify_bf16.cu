// verify_bf16.cu — gdn_verify instantiations for bf16 qkv / conv / out.
#include "verify_impl.cuh"

namespace gdn {
cudaError_t launch_verify_bf16(const VerifyArgs& a, const CUtensorMap& smap, int D, bool tree,
                               cudaStream_t s) {
    return tree ? launch_verify_io<__nv_bfloat16, true>(a, smap, D, s)
                : launch_verify_io<__nv_bfloat16, false>(a, smap, D, s);
}
}  // namespace gdn
