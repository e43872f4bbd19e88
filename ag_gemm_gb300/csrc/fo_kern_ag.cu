// Kernel instantiations: AG-GEMM (bf16 out) with W as [K x N] or [N x K],
// single CTA or CTA pair, without or with gather-buffer movers, or with the
// gather buffers written from the loaded operand stages.
#include "fo_launch.cuh"

cudaError_t fo_variant_ag(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas) {
  switch (v) {
    case FO_V_AG_BF16_KN: return FO_DISPATCH_PAIR(fo::EPI_AG, false, true, false);
    case FO_V_AG_BF16_NK: return FO_DISPATCH_PAIR(fo::EPI_AG, false, false, false);
    case FO_V_AG_BF16_KN_MOV: return FO_DISPATCH_PAIR_MOV(fo::EPI_AG, false, true, false);
    case FO_V_AG_BF16_NK_MOV: return FO_DISPATCH_PAIR_MOV(fo::EPI_AG, false, false, false);
    case FO_V_AG_BF16_KN_GST: return FO_DISPATCH_PAIR_GST(fo::EPI_AG, false, true, false);
    case FO_V_AG_BF16_NK_GST: return FO_DISPATCH_PAIR_GST(fo::EPI_AG, false, false, false);
  }
  return cudaErrorInvalidValue;
}
