// verify_bf16.cu — gdn_verify instantiations for bf16 qkv / conv / out, and the fused
// rollback + verify of the pipelined kernel.
#include "verify_pipe.cuh"

namespace gdn {
cudaError_t launch_verify_bf16(const VerifyArgs& a, const VerifyMaps& m, int D, bool tree,
                               cudaStream_t s) {
    if (verify_pipe_eligible<__nv_bfloat16>(a, m, D, tree, false))
        return launch_verify_pipe<__nv_bfloat16, false>(a, m, tree, s);
    return tree ? launch_verify_io<__nv_bfloat16, true>(a, m.state, D, s)
                : launch_verify_io<__nv_bfloat16, false>(a, m.state, D, s);
}

cudaError_t launch_rollback_verify_bf16(const VerifyArgs& a, const VerifyMaps& m, int D,
                                        cudaStream_t s) {
    if (!verify_pipe_eligible<__nv_bfloat16>(a, m, D, false, true)) return cudaErrorNotSupported;
    return launch_verify_pipe<__nv_bfloat16, true>(a, m, false, s);
}
}  // namespace gdn
