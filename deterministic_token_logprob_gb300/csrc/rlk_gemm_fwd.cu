// rlk_gemm_fwd.cu -- instantiations of the tile engine for the forward: MODE_FWD, and
// MODE_FWDP (the same kernel that also saves bf16 probabilities), see rlk_gemm.cuh.
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_fwd(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                            cudaStream_t stream) {
  if (a.p_out) return launch_gemm<MODE_FWDP>(tmA, tmB, a, stream);
  return launch_gemm<MODE_FWD>(tmA, tmB, a, stream);
}

}  // namespace rlk
