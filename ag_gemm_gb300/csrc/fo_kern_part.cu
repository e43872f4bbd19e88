// Kernel instantiations: pure-GEMM control of GEMM-RS (partials stored into
// the computing rank's own buffer, no transfer).
#include "fo_launch.cuh"

cudaError_t fo_variant_part(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas) {
  switch (v) {
    case FO_V_PART_BF16_KN: return FO_DISPATCH_PAIR(fo::EPI_PARTIAL, false, true, false);
    case FO_V_PART_BF16_NK: return FO_DISPATCH_PAIR(fo::EPI_PARTIAL, false, false, false);
    case FO_V_PART_TF32_NK: return FO_DISPATCH_SINGLE(fo::EPI_PARTIAL, false, false, true);
  }
  return cudaErrorInvalidValue;
}
