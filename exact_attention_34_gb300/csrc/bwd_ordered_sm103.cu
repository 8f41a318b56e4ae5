// Single-pass backward with dQ added in key-tile order (bitwise
// reproducible): the instances of the ordered build of the kernel in
// bwd_single_pass.cuh, compiled apart from the atomic build.
#include "bwd_single_pass.cuh"

namespace attn {
namespace bwd {

template <int D>
cudaError_t launch_single_pass_ordered(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                       const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                       const BwdKParams& kp, dim3 grid, long n_dq, bool f16, cudaStream_t stream) {
  return launch_single_pass_build<D, true>(tq, tk, tv, tdo, tdk, tdv, kp, grid, n_dq, f16, stream);
}

template cudaError_t launch_single_pass_ordered<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                    const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                    const BwdKParams&, dim3, long, bool, cudaStream_t);
template cudaError_t launch_single_pass_ordered<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const BwdKParams&, dim3, long, bool, cudaStream_t);

}  // namespace bwd
}  // namespace attn
