// rlk_gemm_fwd.cu -- instantiation of the tile engine for MODE_FWD (see rlk_gemm.cuh).
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_fwd(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                           cudaStream_t stream) {
  return launch_gemm<MODE_FWD>(tmA, tmB, a, stream);
}

}  // namespace rlk
