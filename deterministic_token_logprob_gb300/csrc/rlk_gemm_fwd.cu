// rlk_gemm_fwd.cu -- instantiations of the tile engine for the forward: MODE_FWD, and
// MODE_FWDP (the same kernel that also saves bf16 probabilities), see rlk_gemm.cuh.
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_fwd(const TileMaps& maps, const GemmArgs& a,
                            cudaStream_t stream) {
  if (a.p_out) return launch_gemm<MODE_FWDP>(maps, a, stream);
  return launch_gemm<MODE_FWD>(maps, a, stream);
}

}  // namespace rlk
