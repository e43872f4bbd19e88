// Kernel instantiations: DP weight gradient (both operands MN-major), fused
// reduce-scatter and its pure-GEMM control, single CTA or CTA pair.
#include "fo_launch.cuh"

cudaError_t fo_variant_dp(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas) {
  switch (v) {
    case FO_V_DP_BF16: return FO_DISPATCH_PAIR(fo::EPI_RS, true, true, false);
    case FO_V_PART_DP: return FO_DISPATCH_PAIR(fo::EPI_PARTIAL, true, true, false);
  }
  return cudaErrorInvalidValue;
}
