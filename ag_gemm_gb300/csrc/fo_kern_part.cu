// Kernel instantiations: pure-GEMM control of GEMM-RS (partials stored into
// the computing rank's own buffer, no transfer).
#include "fo_launch.cuh"

cudaError_t fo_launch_part(int v, const fo::FoParams& p, int grid, cudaStream_t s) {
  switch (v) {
    case FO_V_PART_BF16_KN: return fo_launch_one<fo::EPI_PARTIAL, false, true, false>(p, grid, s);
    case FO_V_PART_BF16_NK: return fo_launch_one<fo::EPI_PARTIAL, false, false, false>(p, grid, s);
    case FO_V_PART_TF32_NK: return fo_launch_one<fo::EPI_PARTIAL, false, false, true>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}
