// Kernel instantiations: AG-GEMM (bf16 out) with W as [K x N] or [N x K].
#include "fo_launch.cuh"

cudaError_t fo_launch_ag(int v, const fo::FoParams& p, int grid, cudaStream_t s) {
  switch (v) {
    case FO_V_AG_BF16_KN: return fo_launch_one<fo::EPI_AG, false, true, false>(p, grid, s);
    case FO_V_AG_BF16_NK: return fo_launch_one<fo::EPI_AG, false, false, false>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}
