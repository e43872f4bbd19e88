// fo_gemm_rs_noalloc: the fused GEMM + reduce-scatter for callers that cannot
// allocate device memory (see include/flashoverlap.h). Same kernel and result
// as fo_gemm_rs; its readiness counters and status word live in a file-scope
// __device__ array instead of a caller-provided workspace.
#include <string.h>

#include <mutex>

#include "fo_internal.h"
#include "fo_kernel.cuh"

// The scratch every fo_gemm_rs_noalloc call uses. In host code this name is
// only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, looked up once per device below.
static __device__ __align__(256) unsigned char g_fo_noalloc_scratch[FO_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set up on the
// first call per device, with that device current).
fo_status scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return FO_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fo_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FO_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FO_OK;
}

}  // namespace

extern "C" fo_status fo_gemm_rs_noalloc(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y,
                                        fo_stream_t stream) {
  // Checks that need only the plan come first, so a plan this entry point
  // cannot run is refused the same way with or without a GPU.
  if (!p || p->d.op != FO_OP_GEMM_RS) return FO_ERR_INVALID_ARG;
  if (p->ring) return FO_ERR_UNSUPPORTED;   // the ring's receive buffers are workspace-sized
  fo_status st;
  if ((st = fo_internal_check_ptrs(p->R, X)) || (st = fo_internal_check_ptrs(p->R, W)) ||
      (st = fo_internal_check_ptrs(p->R, (const void* const*)Y)))
    return st;
  // The tail split's buffers end the workspace; this entry point never
  // splits, so it needs only what comes before them (timestamps of a traced
  // plan included, which alone exceed the array).
  if (p->ws_split_off > (size_t)FO_NOALLOC_SCRATCH_BYTES || p->d.trace) return FO_ERR_SCRATCH_LIMIT;
  if (p->d.out_dtype != FO_F32) return FO_ERR_DTYPE;
  // fp32 W given as [K x N] is transposed into the workspace before the
  // fused launch; this entry point has no room for that copy.
  if (p->elem_bytes == 4 && p->d.w_layout == FO_W_KN) return FO_ERR_UNSUPPORTED;
  if ((st = fo_internal_check_device_ptrs(p->R, X, stream)) || (st = fo_internal_check_device_ptrs(p->R, W, stream)) ||
      (st = fo_internal_check_device_ptrs(p->R, (const void* const*)Y, stream)))
    return st;
  void* scratch = nullptr;
  if ((st = scratch_on_current_device(&scratch))) return st;
  fo::FoParams params;   // on the stack: no host allocation either
  int variant = 0, grid = 0;
  if ((st = fo_internal_rs_params_nocache(p, X, W, Y, scratch, &params, &variant, &grid))) return st;
  // The previous call's counters reset themselves, but a call that timed out
  // leaves them (and the status word) set: start every call from zero.
  if (cudaMemsetAsync(scratch, 0, p->ws_split_off, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  if (fo_launch_variant(variant, p->pair, params, grid, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  p->last_launches = 1;
  return FO_OK;
}
