// Kernel instantiations: DP weight gradient (both operands MN-major), fused
// reduce-scatter and its pure-GEMM control.
#include "fo_launch.cuh"

cudaError_t fo_launch_dp(int v, const fo::FoParams& p, int grid, cudaStream_t s) {
  switch (v) {
    case FO_V_DP_BF16: return fo_launch_one<fo::EPI_RS, true, true, false>(p, grid, s);
    case FO_V_PART_DP: return fo_launch_one<fo::EPI_PARTIAL, true, true, false>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}
