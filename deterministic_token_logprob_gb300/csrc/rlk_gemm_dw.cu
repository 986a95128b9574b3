// rlk_gemm_dw.cu -- instantiation of the tile engine for MODE_DW (see rlk_gemm.cuh).
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_dw(const TileMaps& maps, const GemmArgs& a,
                           cudaStream_t stream) {
  return launch_gemm<MODE_DW>(maps, a, stream);
}

}  // namespace rlk
