// verify_f32.cu — gdn_verify instantiations for fp32 qkv / conv / out.
#include "verify_impl.cuh"

namespace gdn {
cudaError_t launch_verify_f32(const VerifyArgs& a, const VerifyMaps& m, int D, bool tree,
                              cudaStream_t s) {
    return tree ? launch_verify_io<float, true>(a, m.state, D, s)
                : launch_verify_io<float, false>(a, m.state, D, s);
}
}  // namespace gdn
