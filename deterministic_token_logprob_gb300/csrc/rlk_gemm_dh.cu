// rlk_gemm_dh.cu -- instantiation of the tile engine for MODE_DH (see rlk_gemm.cuh).
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_dh(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream) {
  return launch_gemm<MODE_DH>(maps, a, stream);
}

}  // namespace rlk
