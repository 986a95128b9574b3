// rlk_gemm_fp8.cu -- instantiations of the tile engine on E4M3 operands: MODE_FWD8
// (forward statistics) and MODE_DZ8 (the straight-through backward's dz), see rlk_gemm.cuh.
#include "rlk_gemm.cuh"

namespace rlk {

cudaError_t launch_gemm_fwd8(const TileMaps& maps, const GemmArgs& a, cudaStream_t stream) {
  return launch_gemm<MODE_FWD8>(maps, a, stream);
}

cudaError_t launch_gemm_dz8(const TileMaps& maps, const GemmArgs& a, cudaStream_t stream) {
  return launch_gemm<MODE_DZ8>(maps, a, stream);
}

}  // namespace rlk
