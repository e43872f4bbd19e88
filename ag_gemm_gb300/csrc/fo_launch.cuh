// Launch helpers shared by the kernel-instantiation translation units.
#pragma once

#include "fo_kernel.cuh"

template <int EPI, bool A_MN, bool B_MN, bool TF32, bool PAIR, bool MOV = false, bool GST = false, bool SK = false>
cudaError_t fo_launch_one(const fo::FoParams& p, int grid, cudaStream_t stream) {
  auto kern = fo::fo_chunk_gemm_kernel<EPI, A_MN, B_MN, TF32, PAIR, MOV, GST, SK>;
  constexpr int smem = fo::Cfg<PAIR, SK>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(fo::threads_for(MOV));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if constexpr (PAIR) {
    // Clusters of two CTAs; the grid never exceeds the clusters that fit on
    // the device at once (fo_max_ctas_one), so every pair is resident.
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    // Cooperative: every CTA is resident at once, which the cross-CTA
    // readiness waits rely on (a CTA only waits for tiles that come earlier
    // in the static order, so co-residency rules out deadlock).
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int EPI, bool A_MN, bool B_MN, bool TF32, bool PAIR, bool MOV = false, bool GST = false, bool SK = false>
cudaError_t fo_max_ctas_one(int* ctas) {
  auto kern = fo::fo_chunk_gemm_kernel<EPI, A_MN, B_MN, TF32, PAIR, MOV, GST, SK>;
  constexpr int smem = fo::Cfg<PAIR, SK>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * sms));
    cfg.blockDim = dim3(fo::threads_for(MOV));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg)) != cudaSuccess) return e;
    *ctas = 2 * clusters;
  } else {
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, fo::threads_for(MOV), smem)) != cudaSuccess)
      return e;
    *ctas = per_sm * sms;
  }
  return cudaSuccess;
}

// One variant in both tile configurations: launch or size.
#define FO_DISPATCH_PAIR(EPI, A_MN, B_MN, TF32)                                              \
  (pair ? (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, true>(ctas)                          \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, true>(*p, grid, s))                     \
        : (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, false>(ctas)                         \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, false>(*p, grid, s)))
// The short-reduction variant: CTA pairs only.
#define FO_DISPATCH_PAIR_SK(EPI, A_MN, B_MN, TF32)                                           \
  (pair ? (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, true, false, false, true>(ctas)      \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, true, false, false, true>(*p, grid, s)) \
        : cudaErrorInvalidValue)
#define FO_DISPATCH_SINGLE(EPI, A_MN, B_MN, TF32)                                            \
  (pair ? cudaErrorInvalidValue                                                               \
        : (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, false>(ctas)                         \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, false>(*p, grid, s)))
#define FO_DISPATCH_PAIR_MOV(EPI, A_MN, B_MN, TF32)                                          \
  (pair ? (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, true, true>(ctas)                    \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, true, true>(*p, grid, s))               \
        : (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, false, true>(ctas)                   \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, false, true>(*p, grid, s)))
#define FO_DISPATCH_PAIR_GST(EPI, A_MN, B_MN, TF32)                                          \
  (pair ? (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, true, false, true>(ctas)             \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, true, false, true>(*p, grid, s))        \
        : (ctas ? fo_max_ctas_one<EPI, A_MN, B_MN, TF32, false, false, true>(ctas)            \
                : fo_launch_one<EPI, A_MN, B_MN, TF32, false, false, true>(*p, grid, s)))
