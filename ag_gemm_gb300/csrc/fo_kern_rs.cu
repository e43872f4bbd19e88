// Kernel instantiations: GEMM-RS (bf16 with W as [K x N] or [N x K]; fp32
// inputs on the tf32 MMA with W as [N x K]).
#include "fo_launch.cuh"

cudaError_t fo_launch_rs(int v, const fo::FoParams& p, int grid, cudaStream_t s) {
  switch (v) {
    case FO_V_RS_BF16_KN: return fo_launch_one<fo::EPI_RS, false, true, false>(p, grid, s);
    case FO_V_RS_BF16_NK: return fo_launch_one<fo::EPI_RS, false, false, false>(p, grid, s);
    case FO_V_RS_TF32_NK: return fo_launch_one<fo::EPI_RS, false, false, true>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}
