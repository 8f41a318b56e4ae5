// Single-pass backward with atomic dQ adds (not bitwise reproducible), and
// the entry point of both single-pass builds; the kernel is in
// bwd_single_pass.cuh, the ordered build's instances in bwd_ordered_sm103.cu.
#include "bwd_single_pass.cuh"

namespace attn {
namespace bwd {

template <int D>
cudaError_t launch_single_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                               const BwdKParams& kp, dim3 grid, long n_dq, bool f16, bool ordered,
                               cudaStream_t stream) {
  if (ordered) return launch_single_pass_ordered<D>(tq, tk, tv, tdo, tdk, tdv, kp, grid, n_dq, f16, stream);
  return launch_single_pass_build<D, false>(tq, tk, tv, tdo, tdk, tdv, kp, grid, n_dq, f16, stream);
}

template cudaError_t launch_single_pass<64>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                            const BwdKParams&, dim3, long, bool, bool, cudaStream_t);
template cudaError_t launch_single_pass<128>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                             const BwdKParams&, dim3, long, bool, bool, cudaStream_t);

}  // namespace bwd
}  // namespace attn
