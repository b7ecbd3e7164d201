// verify_bf16.cu — gdn_verify instantiations for bf16 qkv / conv / out.
#include "verify_pipe.cuh"

namespace gdn {
cudaError_t launch_verify_bf16(const VerifyArgs& a, const CUtensorMap& smap, int D, bool tree,
                               cudaStream_t s) {
    if (verify_pipe_eligible<__nv_bfloat16>(a, D, tree)) return launch_verify_pipe<__nv_bfloat16>(a, smap, s);
    return tree ? launch_verify_io<__nv_bfloat16, true>(a, smap, D, s)
                : launch_verify_io<__nv_bfloat16, false>(a, smap, D, s);
}
}  // namespace gdn
