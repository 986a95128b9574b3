// rlk_gemm_dz.cu -- instantiation of the tile engine for MODE_DZ (see rlk_gemm.cuh).
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_dz(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                           cudaStream_t stream) {
  return launch_gemm<MODE_DZ>(tmA, tmB, a, stream);
}

}  // namespace rlk
