// Kernel instantiations: GEMM-RS (bf16 with W as [K x N] or [N x K], single
// CTA or CTA pair; fp32 inputs on the tf32 MMA with W as [N x K], single CTA).
#include "fo_launch.cuh"

// Launch (ctas == nullptr) or report the resident-CTA limit of a variant.
cudaError_t fo_variant_rs(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas) {
  switch (v) {
    case FO_V_RS_BF16_KN: return FO_DISPATCH_PAIR(fo::EPI_RS, false, true, false);
    case FO_V_RS_BF16_NK: return FO_DISPATCH_PAIR(fo::EPI_RS, false, false, false);
    case FO_V_RS_TF32_NK: return FO_DISPATCH_SINGLE(fo::EPI_RS, false, false, true);
    case FO_V_RS_BF16_KN_SK: return FO_DISPATCH_PAIR_SK(fo::EPI_RS, false, true, false);
  }
  return cudaErrorInvalidValue;
}
