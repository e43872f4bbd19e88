// Launch helper shared by the kernel-instantiation translation units.
#pragma once

#include "fo_kernel.cuh"

template <int EPI, bool A_MN, bool B_MN, bool TF32>
cudaError_t fo_launch_one(const fo::FoParams& p, int grid, cudaStream_t stream) {
  auto kern = fo::fo_chunk_gemm_kernel<EPI, A_MN, B_MN, TF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fo::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(fo::kThreads);
  cfg.dynamicSmemBytes = fo::kSmemBytes;
  cfg.stream = stream;
  // Cooperative: every CTA is resident at once, which the cross-CTA
  // readiness waits rely on (a CTA only waits for tiles that come earlier in
  // the static order, so co-residency rules out deadlock).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
