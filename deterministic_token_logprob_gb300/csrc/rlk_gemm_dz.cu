// rlk_gemm_dz.cu -- instantiation of the tile engine for MODE_DZ (see rlk_gemm.cuh).
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_dz(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream) {
  return launch_gemm<MODE_DZ>(maps, a, stream);
}

}  // namespace rlk
