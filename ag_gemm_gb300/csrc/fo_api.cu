// C ABI of libflashoverlap.so: argument checks, TMA descriptor encoding,
// launches of the persistent chunk-GEMM kernel and of the two auxiliary
// kernels used by the unfused baselines, and the device status query.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "fo_internal.h"
#include "fo_kernel.cuh"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

struct DevInfo {
  int sms = 0;
  bool sm103 = false;
};

// Per-device properties, queried once per device.
fo_status device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FO_ERR_CUDA;
    }
    cache[dev].sms = sms;
    cache[dev].sm103 = (major == 10 && minor == 3);
    have[dev] = true;
  }
  *out = cache[dev];
  return FO_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool enc2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner, uint64_t outer,
           uint64_t row_bytes, uint32_t box_in, uint32_t box_out) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool enc3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
           uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1_bytes, s2_bytes};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Kernel variant of a GEMM-RS / GEMM-AR plan: bf16 operands with W as
// [K x N] (B MN-major) or [N x K] (B K-major); tf32 operands always with B
// K-major (a W given as [K x N] is first transposed into the workspace).
// A direct reduce-scatter over CTA pairs with at most 12 k-blocks a task
// (K_r <= 768) runs the short-reduction variant: one pipeline stage fewer,
// twice the epilogue's staging buffers. On the attention projection
// (K_r = 512, fp32 out) that took 0.351 ms to 0.320 ms; on the
// 8192 x 1792 x 4096 reduce-scatter (28 k-blocks) the same split cost 6%.
int rs_variant(fo_plan_t p) {
  if (p->elem_bytes == 4) return FO_V_RS_TF32_NK;
  if (p->d.w_layout == FO_W_KN && p->pair && p->num_kb <= 12 && p->d.op == FO_OP_GEMM_RS && !p->ring)
    return FO_V_RS_BF16_KN_SK;
  return p->d.w_layout == FO_W_KN ? FO_V_RS_BF16_KN : FO_V_RS_BF16_NK;
}

// fp32 W_r given as [K_r x N]: the tf32 MMA takes both operands K-major,
// so every call first writes W_r^T [N x K_r] into the workspace.
bool tf32_kn(fo_plan_t p) { return p->elem_bytes == 4 && p->d.w_layout == FO_W_KN; }
float* wt_copy(fo_plan_t p, void* ws, int r) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + p->ws_wt_off + (size_t)r * p->ws_wt_stride);
}

enum CallKind { KIND_NONE = 0, KIND_RS = 1, KIND_DP = 2, KIND_AG = 3, KIND_PART = 4, KIND_A2A = 5, KIND_PART_SHARDED = 6 };

// Returns the cached parameter block when the same call kind is made with
// the same pointers again, else nullptr.
fo::FoParams* cached_params(fo_plan_t p, int kind, const void* const* a, const void* const* b,
                            const void* const* d, const void* const* g = nullptr) {
  if (!p->param_cache || p->param_cache_kind != kind) return nullptr;
  for (int r = 0; r < p->R; ++r)
    if (p->param_cache_key[r] != a[r] || p->param_cache_key[FO_MAX_R + r] != b[r] ||
        p->param_cache_key[2 * FO_MAX_R + r] != d[r] || p->param_cache_key[3 * FO_MAX_R + r] != (g ? g[r] : nullptr))
      return nullptr;
  return static_cast<fo::FoParams*>(p->param_cache);
}

fo::FoParams* fresh_params(fo_plan_t p) {
  if (!p->param_cache) {
    void* mem = nullptr;
    if (posix_memalign(&mem, 128, sizeof(fo::FoParams))) return nullptr;
    p->param_cache = mem;
  }
  p->param_cache_kind = KIND_NONE;
  memset(p->param_cache, 0, sizeof(fo::FoParams));
  return static_cast<fo::FoParams*>(p->param_cache);
}

void remember(fo_plan_t p, int kind, const void* const* a, const void* const* b, const void* const* d,
              const void* const* g = nullptr) {
  for (int r = 0; r < p->R; ++r) {
    p->param_cache_key[r] = a[r];
    p->param_cache_key[FO_MAX_R + r] = b[r];
    p->param_cache_key[2 * FO_MAX_R + r] = d[r];
    p->param_cache_key[3 * FO_MAX_R + r] = g ? g[r] : nullptr;
  }
  p->param_cache_kind = kind;
}

void fill_common(fo_plan_t p, fo::FoParams* k, void* ws) {
  memcpy(k->table, p->table, sizeof(k->table));
  memcpy(k->ord, p->ord, sizeof(k->ord));
  memcpy(k->task_r, p->task_r, sizeof(k->task_r));
  memcpy(k->task_s, p->task_s, sizeof(k->task_s));
  k->R = p->R;
  k->tiles_m = p->tiles_m;
  k->ctr_tiles_m = p->ctr_tiles_m;
  k->tiles_n = p->tiles_n;
  k->num_kb = p->num_kb;
  k->rows_per_chunk = (int32_t)p->rows_per_chunk;
  k->deterministic = p->d.deterministic ? 1 : 0;
  k->fault_inject = p->d.fault_inject;
  k->counters = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + p->ws_counters_off);
  k->status = static_cast<int32_t*>(ws);
  k->timeout_ns = p->d.timeout_ns;
  k->flags = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + p->ws_flags_off);
  k->epoch = &static_cast<fo_ws_header*>(ws)->epoch;
  k->pieces = p->pieces;
  k->row_bytes = p->d.K * 2;
  k->ag_copy = p->d.op == FO_OP_AG_GEMM && p->d.ag_transport == FO_AG_COPY ? 1 : 0;
  k->a2a = p->d.op == FO_OP_GEMM_A2A ? 1 : 0;
  k->n_cols = p->n_out;
  k->trace = p->d.trace ? reinterpret_cast<uint64_t*>(static_cast<char*>(ws) + p->ws_trace_off) : nullptr;
  // Tail split: decided per launch (run_chunk_gemm) once the grid is known.
  k->sk_tiles = 0;
  if (p->sk_cap) {
    float* buf = reinterpret_cast<float*>(static_cast<char*>(ws) + p->ws_split_off);
    if (k->sk_buf != buf) {
      const uint64_t rows = (uint64_t)p->sk_cap * (p->pair ? 2 * FO_BM : FO_BM);
      if (!enc2d(&k->tmSK, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, buf, FO_BN, rows, FO_BN * 4, 32, 32)) buf = nullptr;
    }
    k->sk_buf = buf;
    k->sk_ctr = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + p->ws_split_ctr_off);
  }
  k->delay_ns = p->d.fault_inject == FO_INJECT_DELAY_FIRST_TASK ? (uint64_t)p->d.inject_delay_us * 1000ull : 0ull;
}

fo_status check_ptrs(int R, const void* const* a) {
  if (!a) return FO_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r) {
    if (!a[r]) return FO_ERR_INVALID_ARG;
    if (!aligned16(a[r])) return FO_ERR_ALIGN;
  }
  return FO_OK;
}

// Every pointer must address memory the current device can read and write
// at that same address: its own device memory, managed memory, or host
// memory pinned or registered with CUDA (mapped into the unified address
// space). Pageable host memory and another GPU's memory are rejected, so a
// wrong pointer fails here instead of faulting in the kernel. The query is
// skipped while `stream` captures a graph, and for pointers the driver cannot
// classify.
fo_status check_device_ptrs(int R, const void* const* a, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return FO_OK;
  }
  if (cs != cudaStreamCaptureStatusNone) return FO_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return FO_OK;
  }
  for (int r = 0; r < R; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, a[r]) != cudaSuccess) {
      cudaGetLastError();
      continue;
    }
    switch (at.type) {
      case cudaMemoryTypeDevice:
        if (at.device != dev) return FO_ERR_INVALID_ARG;
        break;
      case cudaMemoryTypeManaged:
        break;
      case cudaMemoryTypeHost:
        if (at.devicePointer != a[r]) return FO_ERR_INVALID_ARG;
        break;
      default:   // pageable host memory
        return FO_ERR_INVALID_ARG;
    }
  }
  return FO_OK;
}

// The same for every pointer a call hands the kernel (G and ws may be null).
fo_status check_call_ptrs(int R, const void* const* a, const void* const* b, const void* const* d,
                          const void* const* g, const void* ws, cudaStream_t s) {
  fo_status st;
  if ((st = check_device_ptrs(R, a, s)) || (st = check_device_ptrs(R, b, s)) || (st = check_device_ptrs(R, d, s)))
    return st;
  if (g && (st = check_device_ptrs(R, g, s))) return st;
  if (ws && (st = check_device_ptrs(1, &ws, s))) return st;
  return FO_OK;
}

// Encode the operand maps of a GEMM-RS / DP-grad-RS / GEMM-AR / pure-control
// call. The fp32 destination of the partials is: Y_c (RS/DP with fp32 out),
// the workspace's shard sums (bf16 out), rank c's own rows of its full
// output (AR), or the computing rank's own buffer (partials control). Under
// the ring RS the forwards go to the receivers' buffers in the workspace and
// only the last hop writes Y_c.
fo_status build_rs_like(fo_plan_t p, bool dp, bool partial, const void* const* A, const void* const* B,
                        void* const* D, void* ws, cudaStream_t stream, fo::FoParams** out) {
  const int kind = partial ? KIND_PART : (dp ? KIND_DP : KIND_RS);
  const bool ring = !partial && p->ring;
  const bool bf16_out = !partial && p->d.out_dtype == FO_BF16;
  const bool to_ws = bf16_out && !ring;
  const bool ar = !partial && p->d.op == FO_OP_GEMM_AR;
  const bool wt = !dp && tf32_kn(p);
  fo::FoParams* k = cached_params(p, kind, A, B, (const void* const*)D);
  if (k && ((!to_ws && !ring && !wt) || p->param_cache_ws == ws)) {
    fill_common(p, k, ws);
    *out = k;
    return FO_OK;
  }
  if (fo_status st = check_call_ptrs(p->R, A, B, (const void* const*)D, nullptr, ws, stream)) return st;
  k = fresh_params(p);
  if (!k) return FO_ERR_INVALID_ARG;
  const int R = p->R;
  const uint64_t M = (uint64_t)p->d.M, N = (uint64_t)p->n_out, rpc = (uint64_t)p->rows_per_chunk;
  const uint64_t kr = (uint64_t)p->k_red;
  const int es = p->elem_bytes;
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint32_t bk = FO_BK_BYTES / es;
  bool ok = true;
  for (int r = 0; r < R && ok; ++r) {
    if (!dp) {
      ok &= enc2d(&k->tmA[r], dt, A[r], kr, M, kr * es, bk, FO_BM);
      if (wt) ok &= enc2d(&k->tmB[r], dt, wt_copy(p, ws, r), kr, N, kr * es, bk, p->pair ? FO_BN / 2 : FO_BN);
      else if (p->d.w_layout == FO_W_KN) ok &= enc2d(&k->tmB[r], dt, B[r], N, kr, N * es, bk, bk);
      else ok &= enc2d(&k->tmB[r], dt, B[r], kr, N, kr * es, bk, p->pair ? FO_BN / 2 : FO_BN);
    } else {
      ok &= enc2d(&k->tmA[r], dt, A[r], M, kr, M * es, bk, bk);
      ok &= enc2d(&k->tmB[r], dt, B[r], N, kr, N * es, bk, bk);
    }
    if (partial) {
      ok &= enc3d(&k->tmD[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D[r], N, rpc, R, N * 4, rpc * N * 4, 32, 32);
      continue;
    }
    float* shard = static_cast<float*>(D[r]);
    if (to_ws) shard = reinterpret_cast<float*>(static_cast<char*>(ws) + p->ws_shard_off + r * p->ws_shard_stride);
    if (ar) shard = static_cast<float*>(D[r]) + (size_t)r * rpc * N;
    if (ring && bf16_out) shard = nullptr;   // the last hop writes the bf16 output directly
    if (shard) ok &= enc2d(&k->tmD[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, shard, N, rpc, N * 4, 32, 32);
    k->shard[r] = shard;
    // The finisher's outputs: the bf16 shard, or every rank's full output
    // viewed as [N, rows/R, R] so a store clips at the shard's last row.
    if (bf16_out) ok &= enc2d(&k->tmF[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D[r], N, rpc, N * 2, 64, 32);
    if (ar) ok &= enc3d(&k->tmAR[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, D[r], N, rpc, R, N * 4, rpc * N * 4, 32, 32);
    if (ring) {
      // Rank r's receive buffer: chunk c's rows at c * rows/R, viewed as
      // [N, rows/R, R] like an all-reduce output.
      float* inbox = reinterpret_cast<float*>(static_cast<char*>(ws) + p->ws_ring_off + r * p->ws_ring_stride);
      k->inbox[r] = inbox;
      ok &= enc3d(&k->tmAR[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, inbox, N, rpc, R, N * 4, rpc * N * 4, 32, 32);
    }
  }
  if (!ok) return FO_ERR_CUDA;
  remember(p, kind, A, B, (const void* const*)D);
  p->param_cache_ws = ws;
  fill_common(p, k, ws);
  k->completion = partial ? fo::FO_COMPLETE_NONE
                          : (bf16_out ? fo::FO_COMPLETE_BF16 : (ar ? fo::FO_COMPLETE_ALLREDUCE : fo::FO_COMPLETE_NONE));
  k->ring = ring ? 1 : 0;
  *out = k;
  return FO_OK;
}

// How an AG call under peer read fills the gather buffers G_r. The mover
// warps copy R*R shards (R*M*K*2 bytes) while the GEMM runs; they keep up
// only while the GEMM is long enough, i.e. for wide outputs. For narrow ones
// (N/R <= 1024 columns) the producer writes each A stage it loaded for the
// first column block into G_r: no extra reads, at the cost of a wait for each
// store before its stage is refilled. Measured on GB300 (R = 8, 8192 x 4096
// gathered): N/R = 512: movers 392 us, stores 282 us (GEMM alone 159 us);
// N/R = 1536: movers 500 us, stores 610 us (GEMM alone 438 us).
bool gather_by_stores(fo_plan_t p) {
  return p->d.ag_transport == FO_AG_PEER_READ && p->n_out <= 1024;
}

fo_status build_ag(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* const* G,
                   void* ws, cudaStream_t stream, fo::FoParams** out) {
  fo::FoParams* k = cached_params(p, KIND_AG, X, W, (const void* const*)Y, (const void* const*)G);
  if (k) {
    fill_common(p, k, ws);
    *out = k;
    return FO_OK;
  }
  if (fo_status st = check_call_ptrs(p->R, X, W, (const void* const*)Y, (const void* const*)G, ws, stream))
    return st;
  k = fresh_params(p);
  if (!k) return FO_ERR_INVALID_ARG;
  const int R = p->R;
  const uint64_t K = (uint64_t)p->d.K, nr = (uint64_t)p->n_out, rpc = (uint64_t)p->rows_per_chunk;
  const uint64_t M = (uint64_t)p->d.M;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok = true;
  for (int r = 0; r < R && ok; ++r) {
    ok &= enc2d(&k->tmA[r], dt, X[r], K, rpc, K * 2, 64, FO_BM);
    if (p->d.w_layout == FO_W_KN) ok &= enc2d(&k->tmB[r], dt, W[r], nr, K, nr * 2, 64, 64);
    else ok &= enc2d(&k->tmB[r], dt, W[r], K, nr, K * 2, 64, p->pair ? FO_BN / 2 : FO_BN);
    ok &= enc3d(&k->tmD[r], dt, Y[r], nr, rpc, R, nr * 2, rpc * nr * 2, 64, 32);
    if (G && gather_by_stores(p)) {
      // G_r is written from the A stages the GEMM loads, viewed as
      // [K, rows/R, R] so that a store clips at the shard's last row.
      ok &= enc3d(&k->tmG[r], dt, G[r], K, rpc, R, K * 2, rpc * K * 2, 64, FO_BM);
    } else if (G) {
      ok &= enc2d(&k->tmG[r], dt, G[r], K, M, K * 2, 64, FO_BM);
      k->xsrc[r] = X[r];
      k->gdst[r] = G[r];
    }
  }
  if (!ok) return FO_ERR_CUDA;
  remember(p, KIND_AG, X, W, (const void* const*)Y, (const void* const*)G);
  fill_common(p, k, ws);
  *out = k;
  return FO_OK;
}

// All-to-all: X_r [M/R x K] as the A operand (like an all-gather shard), the
// whole W_r [K x N] (or [N x K]) as B, read at column block c of each task,
// and each Y_c [M x N/R] viewed [N/R, M/R, R] so that a store of rank r's
// rows clips at its block's last row and column.
fo_status build_a2a(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* ws,
                    cudaStream_t stream, fo::FoParams** out) {
  fo::FoParams* k = cached_params(p, KIND_A2A, X, W, (const void* const*)Y);
  if (k) {
    fill_common(p, k, ws);
    *out = k;
    return FO_OK;
  }
  if (fo_status st = check_call_ptrs(p->R, X, W, (const void* const*)Y, nullptr, ws, stream)) return st;
  k = fresh_params(p);
  if (!k) return FO_ERR_INVALID_ARG;
  const int R = p->R;
  const uint64_t K = (uint64_t)p->d.K, N = (uint64_t)p->d.N, nc = (uint64_t)p->n_out;
  const uint64_t rpc = (uint64_t)p->rows_per_chunk;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  bool ok = true;
  for (int r = 0; r < R && ok; ++r) {
    ok &= enc2d(&k->tmA[r], dt, X[r], K, rpc, K * 2, 64, FO_BM);
    if (p->d.w_layout == FO_W_KN) ok &= enc2d(&k->tmB[r], dt, W[r], N, K, N * 2, 64, 64);
    else ok &= enc2d(&k->tmB[r], dt, W[r], K, N, K * 2, 64, p->pair ? FO_BN / 2 : FO_BN);
    ok &= enc3d(&k->tmD[r], dt, Y[r], nc, rpc, R, nc * 2, rpc * nc * 2, 64, 32);
  }
  if (!ok) return FO_ERR_CUDA;
  remember(p, KIND_A2A, X, W, (const void* const*)Y);
  fill_common(p, k, ws);
  *out = k;
  return FO_OK;
}

fo_status preflight(fo_plan_t p, DevInfo* di) {
  if (!load_encode()) return FO_ERR_CUDA;
  fo_status st = device_info(di);
  if (st != FO_OK) return st;
  if (!di->sm103) return FO_ERR_UNSUPPORTED;
  (void)p;
  return FO_OK;
}

// Launch grid for a plan: single-CTA tiles use min(tiles, resident CTAs);
// pair tiles use an even number of CTAs, at most the pairs resident at once.
fo_status launch_grid(fo_plan_t p, int variant, const DevInfo& di, int* grid) {
  static std::mutex mu;
  static int cache[64][FO_V_COUNT][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  int cap = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    cap = cache[dev][variant][p->pair ? 1 : 0];
  }
  if (cap <= 0) {
    if (fo_max_resident_ctas(variant, p->pair, &cap) != cudaSuccess || cap <= 0) {
      cudaGetLastError();
      return FO_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[dev][variant][p->pair ? 1 : 0] = cap;
  }
  const int total = p->R * p->R * p->tiles_m * p->tiles_n;
  if (p->pair) {
    const int units = total < cap / 2 ? total : cap / 2;
    *grid = 2 * units;
  } else {
    int g = total < di.sms ? total : di.sms;
    *grid = g < cap ? g : cap;
  }
  return *grid > 0 ? FO_OK : FO_ERR_CUDA;
}

fo_status run_chunk_gemm(fo_plan_t p, int variant, fo::FoParams* k, const DevInfo& di, cudaStream_t s) {
  int grid = 0;
  fo_status st = launch_grid(p, variant, di, &grid);
  if (st != FO_OK) return st;
  // Tail split for this launch's units, when the workspace has room for it.
  k->sk_tiles = 0;
  if (p->sk_cap && k->sk_buf) {
    const int sk = fo_tail_split_tiles((int64_t)p->R * p->R * p->tiles_m * p->tiles_n, p->pair ? grid / 2 : grid);
    if (sk <= p->sk_cap) k->sk_tiles = sk;
  }
  cudaError_t e = fo_launch_variant(variant, p->pair, *k, grid, s);
  if (fo_log_enabled())
    fprintf(stderr, "[flashoverlap] launch variant %d, %d CTAs (%s), %d tiles split, stream %p: %s\n", variant,
            grid, p->pair ? "CTA pairs" : "single CTAs", k->sk_tiles, (void*)s, cudaGetErrorString(e));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  p->last_launches = 1;
  p->last_grid = grid;
  p->last_split_tiles = k->sk_tiles;
  return FO_OK;
}

fo_status transpose_w(fo_plan_t p, const void* const* W, void* ws, cudaStream_t s);

// GEMM-RS-like launch; with fp32 W_r given as [K x N], the transpose into the
// workspace goes first on the same stream (two launches).
fo_status run_rs_chunk_gemm(fo_plan_t p, const void* const* W, void* ws, int variant, fo::FoParams* k,
                            const DevInfo& di, cudaStream_t s) {
  if (tf32_kn(p)) {
    if (fo_status st = transpose_w(p, W, ws, s)) return st;
  }
  fo_status st = run_chunk_gemm(p, variant, k, di, s);
  if (st == FO_OK && tf32_kn(p)) p->last_launches = 2;
  return st;
}

// ---------------------------------------------------------------- aux kernels

struct PtrArray {
  const void* p[FO_MAX_R];
};
struct MutPtrArray {
  void* p[FO_MAX_R];
};

// Y_d = sum_r P_r[rows of d]: one float4 of one shard per thread and loop trip.
__global__ void reduce_scatter_f32_kernel(PtrArray P, MutPtrArray Y, int R, int64_t shard_vec4) {
  const int64_t total = shard_vec4 * R;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int d = (int)(i / shard_vec4);
    const int64_t j = i - (int64_t)d * shard_vec4;
    float4 acc = reinterpret_cast<const float4*>(P.p[0])[(int64_t)d * shard_vec4 + j];
    for (int r = 1; r < R; ++r) {
      const float4 v = reinterpret_cast<const float4*>(P.p[r])[(int64_t)d * shard_vec4 + j];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4*>(Y.p[d])[j] = acc;
  }
}

// G_r[rows of src] = X_src for every (r, src): 16-byte copies.
__global__ void all_gather_copy_kernel(PtrArray X, MutPtrArray G, int R, int64_t shard_vec16) {
  const int64_t total = shard_vec16 * R * R;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pair = i / shard_vec16;
    const int64_t j = i - pair * shard_vec16;
    const int r = (int)(pair / R), src = (int)(pair - (int64_t)r * R);
    const int4 v = reinterpret_cast<const int4*>(X.p[src])[j];
    reinterpret_cast<int4*>(G.p[r])[(int64_t)src * shard_vec16 + j] = v;
  }
}

// Y_c[r * rows + i, :] = P_r[i, c block] for every (c, r, i): 16-byte copies,
// one per thread and loop trip (P_r [rows x R * nc16 * 8], Y_c [R * rows x
// nc16 * 8], bf16).
__global__ void all_to_all_copy_kernel(PtrArray P, MutPtrArray Y, int R, int64_t rows, int64_t nc16) {
  const int64_t per_block = rows * nc16;   // one (c, r) block
  const int64_t total = per_block * R * R;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = i / per_block;
    const int64_t w = i - blk * per_block;
    const int c = (int)(blk / R), r = (int)(blk - (int64_t)c * R);
    const int64_t row = w / nc16, v = w - row * nc16;
    const int4 x = reinterpret_cast<const int4*>(P.p[r])[row * nc16 * R + (int64_t)c * nc16 + v];
    reinterpret_cast<int4*>(Y.p[c])[((int64_t)r * rows + row) * nc16 + v] = x;
  }
}

// Wt_r = W_r^T for every rank r (blockIdx.z): W_r [K x N] fp32 row-major,
// Wt_r [N x K]; 32 x 32 tiles through shared memory so that both the reads
// and the writes are coalesced.
__global__ void transpose_f32_kernel(PtrArray W, MutPtrArray Wt, int64_t K, int64_t N) {
  __shared__ float tile[32][33];
  const float* src = static_cast<const float*>(W.p[blockIdx.z]);
  float* dst = static_cast<float*>(Wt.p[blockIdx.z]);
  const int64_t n0 = (int64_t)blockIdx.x * 32;
  for (int64_t k0 = (int64_t)blockIdx.y * 32; k0 < K; k0 += (int64_t)gridDim.y * 32) {
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
      const int64_t k = k0 + i, n = n0 + threadIdx.x;
      tile[i][threadIdx.x] = (k < K && n < N) ? src[k * N + n] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
      const int64_t n = n0 + i, k = k0 + threadIdx.x;
      if (n < N && k < K) dst[n * K + k] = tile[threadIdx.x][i];
    }
    __syncthreads();
  }
}

// Launch the transpose of every rank's fp32 W_r into the workspace (plans
// with fp32 inputs and W as [K x N] only).
fo_status transpose_w(fo_plan_t p, const void* const* W, void* ws, cudaStream_t s) {
  PtrArray wa = {};
  MutPtrArray ta = {};
  for (int r = 0; r < p->R; ++r) {
    wa.p[r] = W[r];
    ta.p[r] = wt_copy(p, ws, r);
  }
  const int64_t K = p->k_red, N = p->n_out;
  const int64_t ky = (K + 31) / 32;
  dim3 grid((unsigned)((N + 31) / 32), (unsigned)(ky < 65535 ? ky : 65535), (unsigned)p->R);
  transpose_f32_kernel<<<grid, dim3(32, 8), 0, s>>>(wa, ta, K, N);
  if (cudaGetLastError() != cudaSuccess) return FO_ERR_CUDA;
  return FO_OK;
}

}  // namespace

// Parameters of one fo_gemm_rs launch built into caller storage (no plan
// cache, no allocation), with the readiness counters and status word in
// `scratch`. Used by the allocation-free entry point.
fo_status fo_internal_rs_params_nocache(fo_plan_t p, const void* const* X, const void* const* W,
                                        void* const* Y, void* scratch, fo::FoParams* k, int* variant,
                                        int* grid) {
  if (p->d.op != FO_OP_GEMM_RS || p->d.out_dtype != FO_F32) return FO_ERR_DTYPE;
  if (p->ring) return FO_ERR_UNSUPPORTED;   // the ring's receive buffers do not fit the static scratch
  if (tf32_kn(p)) return FO_ERR_UNSUPPORTED;   // W_r^T would have to live in the static scratch
  DevInfo di;
  fo_status st = preflight(p, &di);
  if (st != FO_OK) return st;
  memset(static_cast<void*>(k), 0, sizeof(*k));
  const int R = p->R;
  const uint64_t M = (uint64_t)p->d.M, N = (uint64_t)p->d.N, rpc = (uint64_t)p->rows_per_chunk;
  const uint64_t kr = (uint64_t)p->k_red;
  const int es = p->elem_bytes;
  const CUtensorMapDataType dt = es == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const uint32_t bk = FO_BK_BYTES / es;
  bool ok = true;
  for (int r = 0; r < R && ok; ++r) {
    ok &= enc2d(&k->tmA[r], dt, X[r], kr, M, kr * es, bk, FO_BM);
    if (p->d.w_layout == FO_W_KN) ok &= enc2d(&k->tmB[r], dt, W[r], N, kr, N * es, bk, bk);
    else ok &= enc2d(&k->tmB[r], dt, W[r], kr, N, kr * es, bk, p->pair ? FO_BN / 2 : FO_BN);
    ok &= enc2d(&k->tmD[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, Y[r], N, rpc, N * 4, 32, 32);
  }
  if (!ok) return FO_ERR_CUDA;
  fill_common(p, k, scratch);
  k->sk_tiles = 0;   // no tail split: its buffers are not in the static scratch
  k->sk_buf = nullptr;
  k->sk_ctr = nullptr;
  *variant = rs_variant(p);
  return launch_grid(p, *variant, di, grid);
}

fo_status fo_internal_check_ptrs(int R, const void* const* a) { return check_ptrs(R, a); }
fo_status fo_internal_check_device_ptrs(int R, const void* const* a, fo_stream_t stream) {
  return check_device_ptrs(R, a, (cudaStream_t)stream);
}

extern "C" {

fo_status fo_check_device_pointers(int32_t n, const void* const* ptrs, fo_stream_t stream) {
  if (n < 0 || (n > 0 && !ptrs)) return FO_ERR_INVALID_ARG;
  return check_device_ptrs(n, ptrs, (cudaStream_t)stream);
}

fo_status fo_trace_query(fo_plan_t p, const void* ws, fo_stream_t stream, uint64_t* stamps, int32_t cap,
                         int32_t* n_ctas) {
  if (!p || !ws || !n_ctas || cap < 0 || (cap > 0 && !stamps)) return FO_ERR_INVALID_ARG;
  if (!p->d.trace || p->last_grid <= 0) return FO_ERR_INVALID_ARG;
  *n_ctas = p->last_grid;
  int m = p->last_grid < FO_TRACE_MAX_CTAS ? p->last_grid : FO_TRACE_MAX_CTAS;
  if (m > cap) m = cap;
  if (m > 0) {
    const char* src = static_cast<const char*>(ws) + p->ws_trace_off;
    if (cudaMemcpyAsync(stamps, src, (size_t)m * FO_TRACE_STAMPS * sizeof(uint64_t), cudaMemcpyDeviceToHost,
                        (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
      cudaGetLastError();
      return FO_ERR_CUDA;
    }
  }
  return FO_OK;
}

fo_status fo_workspace_init(fo_plan_t p, void* ws, fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws, 0, p->ws_bytes, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  return FO_OK;
}

fo_status fo_gemm_rs(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* ws,
                     fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_GEMM_RS) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, W)) || (st = check_ptrs(p->R, (const void* const*)Y)))
    return st;
  if (!aligned16(ws)) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  fo::FoParams* k = nullptr;
  if ((st = build_rs_like(p, false, false, X, W, Y, ws, (cudaStream_t)stream, &k))) return st;
  return run_rs_chunk_gemm(p, W, ws, rs_variant(p), k, di, (cudaStream_t)stream);
}

fo_status fo_gemm_ar(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* ws,
                     fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_GEMM_AR) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, W)) || (st = check_ptrs(p->R, (const void* const*)Y)))
    return st;
  if (!aligned16(ws)) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  fo::FoParams* k = nullptr;
  if ((st = build_rs_like(p, false, false, X, W, Y, ws, (cudaStream_t)stream, &k))) return st;
  return run_rs_chunk_gemm(p, W, ws, rs_variant(p), k, di, (cudaStream_t)stream);
}

fo_status fo_dp_grad_rs(fo_plan_t p, const void* const* X, const void* const* dY, void* const* dW, void* ws,
                        fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_DP_GRAD_RS) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, dY)) || (st = check_ptrs(p->R, (const void* const*)dW)))
    return st;
  if (!aligned16(ws)) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  fo::FoParams* k = nullptr;
  if ((st = build_rs_like(p, true, false, X, dY, dW, ws, (cudaStream_t)stream, &k))) return st;
  return run_chunk_gemm(p, FO_V_DP_BF16, k, di, (cudaStream_t)stream);
}

fo_status fo_ag_gemm(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* const* G,
                     void* ws, fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_AG_GEMM) return FO_ERR_INVALID_ARG;
  if (p->d.ag_transport == FO_AG_COPY && !G) return FO_ERR_INVALID_ARG;   // the ring needs gather buffers
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, W)) || (st = check_ptrs(p->R, (const void* const*)Y)))
    return st;
  if (G && (st = check_ptrs(p->R, (const void* const*)G))) return st;
  if (!aligned16(ws)) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  fo::FoParams* k = nullptr;
  if ((st = build_ag(p, X, W, Y, G, ws, (cudaStream_t)stream, &k))) return st;
  int v;
  const bool kn = p->d.w_layout == FO_W_KN;
  if (G && gather_by_stores(p)) v = kn ? FO_V_AG_BF16_KN_GST : FO_V_AG_BF16_NK_GST;
  else if (G) v = kn ? FO_V_AG_BF16_KN_MOV : FO_V_AG_BF16_NK_MOV;
  else v = kn ? FO_V_AG_BF16_KN : FO_V_AG_BF16_NK;
  return run_chunk_gemm(p, v, k, di, (cudaStream_t)stream);
}

fo_status fo_gemm_a2a(fo_plan_t p, const void* const* X, const void* const* W, void* const* Y, void* ws,
                      fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, W)) || (st = check_ptrs(p->R, (const void* const*)Y)))
    return st;
  if (!aligned16(ws)) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  fo::FoParams* k = nullptr;
  if ((st = build_a2a(p, X, W, Y, ws, (cudaStream_t)stream, &k))) return st;
  return run_chunk_gemm(p, p->d.w_layout == FO_W_KN ? FO_V_AG_BF16_KN : FO_V_AG_BF16_NK, k, di,
                        (cudaStream_t)stream);
}

fo_status fo_gemm_partials_sharded(fo_plan_t p, const void* const* A, const void* const* B, void* const* P,
                                   void* ws, fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_DP_GRAD_RS || p->elem_bytes != 2) return FO_ERR_INVALID_ARG;
  const int R = p->R;
  const uint64_t kr = (uint64_t)p->k_red;                  // T: the reduction, split into R shards of rows
  const uint32_t bk = FO_BK_BYTES / 2;
  if (kr % (uint64_t)R || (kr / (uint64_t)R) % bk) return FO_ERR_SHAPE;   // a k-block never straddles two shards
  fo_status st;
  if ((st = check_ptrs(R, A)) || (st = check_ptrs(R, B)) || (st = check_ptrs(R, (const void* const*)P))) return st;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  const uint64_t M = (uint64_t)p->d.M, N = (uint64_t)p->n_out, rpc = (uint64_t)p->rows_per_chunk;
  // Shards that lie back to back in rank order already form the gathered
  // A: one tensor map over all of it, the same for every rank. Otherwise
  // one map per shard, picked per k-block (measured on GB300 at the
  // layer's 8192 x 4096 shapes: about 4% slower than one map).
  const uint64_t shard_bytes = kr / (uint64_t)R * M * 2;
  bool adjacent = true;
  for (int s = 1; s < R; ++s)
    adjacent &= static_cast<const char*>(A[s]) == static_cast<const char*>(A[0]) + s * shard_bytes;
  fo::FoParams* k = cached_params(p, KIND_PART_SHARDED, A, B, (const void* const*)P);
  if (!k) {
    if ((st = check_call_ptrs(R, A, B, (const void* const*)P, nullptr, ws, (cudaStream_t)stream))) return st;
    k = fresh_params(p);
    if (!k) return FO_ERR_INVALID_ARG;
    bool ok = true;
    for (int r = 0; r < R && ok; ++r) {
      if (adjacent) ok &= enc2d(&k->tmA[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A[0], M, kr, M * 2, bk, bk);
      else ok &= enc2d(&k->tmA[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A[r], M, kr / (uint64_t)R, M * 2, bk, bk);
      ok &= enc2d(&k->tmB[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B[r], N, kr, N * 2, bk, bk);
      ok &= enc3d(&k->tmD[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, P[r], N, rpc, R, N * 4, rpc * N * 4, 32, 32);
    }
    if (!ok) return FO_ERR_CUDA;
    remember(p, KIND_PART_SHARDED, A, B, (const void* const*)P);
    p->param_cache_ws = ws;
  }
  fill_common(p, k, ws);
  k->completion = fo::FO_COMPLETE_NONE;
  k->ring = 0;
  k->a_shard_rows = adjacent ? 0 : (int32_t)(kr / (uint64_t)R);
  return run_chunk_gemm(p, FO_V_PART_DP, k, di, (cudaStream_t)stream);
}

fo_status fo_gemm_partials(fo_plan_t p, const void* const* A, const void* const* B, void* const* P, void* ws,
                           fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op == FO_OP_AG_GEMM || p->d.op == FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, A)) || (st = check_ptrs(p->R, B)) || (st = check_ptrs(p->R, (const void* const*)P)))
    return st;
  DevInfo di;
  if ((st = preflight(p, &di))) return st;
  const bool dp = p->d.op == FO_OP_DP_GRAD_RS;
  fo::FoParams* k = nullptr;
  if ((st = build_rs_like(p, dp, true, A, B, P, ws, (cudaStream_t)stream, &k))) return st;
  int v = dp ? FO_V_PART_DP
             : (p->elem_bytes == 4 ? FO_V_PART_TF32_NK
                                   : (p->d.w_layout == FO_W_KN ? FO_V_PART_BF16_KN : FO_V_PART_BF16_NK));
  if (dp) return run_chunk_gemm(p, v, k, di, (cudaStream_t)stream);
  return run_rs_chunk_gemm(p, B, ws, v, k, di, (cudaStream_t)stream);
}

fo_status fo_reduce_scatter_f32(fo_plan_t p, const void* const* P, void* const* Y, fo_stream_t stream) {
  if (!p) return FO_ERR_INVALID_ARG;
  if (p->d.op == FO_OP_AG_GEMM || p->d.op == FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, P)) || (st = check_ptrs(p->R, (const void* const*)Y))) return st;
  if ((st = check_device_ptrs(p->R, P, (cudaStream_t)stream)) ||
      (st = check_device_ptrs(p->R, (const void* const*)Y, (cudaStream_t)stream)))
    return st;
  if (p->n_out % 4) return FO_ERR_ALIGN;
  DevInfo di;
  if ((st = device_info(&di))) return st;
  PtrArray pa = {};
  MutPtrArray ya = {};
  for (int r = 0; r < p->R; ++r) {
    pa.p[r] = P[r];
    ya.p[r] = Y[r];
  }
  const int64_t shard_vec4 = p->rows_per_chunk * p->n_out / 4;
  reduce_scatter_f32_kernel<<<di.sms * 4, 256, 0, (cudaStream_t)stream>>>(pa, ya, p->R, shard_vec4);
  if (cudaGetLastError() != cudaSuccess) return FO_ERR_CUDA;
  p->last_launches = 1;
  return FO_OK;
}

fo_status fo_all_gather_copy(fo_plan_t p, const void* const* X, void* const* G, fo_stream_t stream) {
  if (!p) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_AG_GEMM) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, X)) || (st = check_ptrs(p->R, (const void* const*)G))) return st;
  if ((st = check_device_ptrs(p->R, X, (cudaStream_t)stream)) ||
      (st = check_device_ptrs(p->R, (const void* const*)G, (cudaStream_t)stream)))
    return st;
  DevInfo di;
  if ((st = device_info(&di))) return st;
  PtrArray xa = {};
  MutPtrArray ga = {};
  for (int r = 0; r < p->R; ++r) {
    xa.p[r] = X[r];
    ga.p[r] = G[r];
  }
  const int64_t shard_vec16 = p->rows_per_chunk * p->d.K * 2 / 16;
  all_gather_copy_kernel<<<di.sms * 4, 256, 0, (cudaStream_t)stream>>>(xa, ga, p->R, shard_vec16);
  if (cudaGetLastError() != cudaSuccess) return FO_ERR_CUDA;
  p->last_launches = 1;
  return FO_OK;
}

fo_status fo_all_to_all_copy(fo_plan_t p, const void* const* P, void* const* Y, fo_stream_t stream) {
  if (!p) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
  fo_status st;
  if ((st = check_ptrs(p->R, P)) || (st = check_ptrs(p->R, (const void* const*)Y))) return st;
  if ((st = check_device_ptrs(p->R, P, (cudaStream_t)stream)) ||
      (st = check_device_ptrs(p->R, (const void* const*)Y, (cudaStream_t)stream)))
    return st;
  DevInfo di;
  if ((st = device_info(&di))) return st;
  PtrArray pa = {};
  MutPtrArray ya = {};
  for (int r = 0; r < p->R; ++r) {
    pa.p[r] = P[r];
    ya.p[r] = Y[r];
  }
  // n_out * 2 bytes is a multiple of 16 (checked by fo_plan).
  all_to_all_copy_kernel<<<di.sms * 4, 256, 0, (cudaStream_t)stream>>>(pa, ya, p->R, p->rows_per_chunk,
                                                                        p->n_out * 2 / 16);
  if (cudaGetLastError() != cudaSuccess) return FO_ERR_CUDA;
  p->last_launches = 1;
  return FO_OK;
}

fo_status fo_status_query(fo_plan_t p, void* ws, fo_stream_t stream, int32_t info[4]) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  int32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  if (info) memcpy(info, h, sizeof(h));
  if (h[0] != 0) {
    if (cudaMemset(ws, 0, p->ws_bytes) != cudaSuccess) {
      cudaGetLastError();
      return FO_ERR_CUDA;
    }
    return (fo_status)h[0];
  }
  return FO_OK;
}

}  // extern "C"

cudaError_t fo_variant_rs(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas);
cudaError_t fo_variant_dp(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas);
cudaError_t fo_variant_ag(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas);
cudaError_t fo_variant_part(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas);

static cudaError_t fo_variant_call(int v, bool pair, const fo::FoParams* p, int grid, cudaStream_t s, int* ctas) {
  switch (v) {
    case FO_V_RS_BF16_KN:
    case FO_V_RS_BF16_NK:
    case FO_V_RS_TF32_NK:
    case FO_V_RS_BF16_KN_SK: return fo_variant_rs(v, pair, p, grid, s, ctas);
    case FO_V_DP_BF16:
    case FO_V_PART_DP: return fo_variant_dp(v, pair, p, grid, s, ctas);
    case FO_V_AG_BF16_KN:
    case FO_V_AG_BF16_NK:
    case FO_V_AG_BF16_KN_MOV:
    case FO_V_AG_BF16_NK_MOV:
    case FO_V_AG_BF16_KN_GST:
    case FO_V_AG_BF16_NK_GST: return fo_variant_ag(v, pair, p, grid, s, ctas);
    case FO_V_PART_BF16_KN:
    case FO_V_PART_BF16_NK:
    case FO_V_PART_TF32_NK: return fo_variant_part(v, pair, p, grid, s, ctas);
  }
  return cudaErrorInvalidValue;
}

cudaError_t fo_launch_variant(int v, bool pair, const fo::FoParams& p, int grid, cudaStream_t s) {
  return fo_variant_call(v, pair, &p, grid, s, nullptr);
}

cudaError_t fo_max_resident_ctas(int v, bool pair, int* ctas) {
  return fo_variant_call(v, pair, nullptr, 0, nullptr, ctas);
}
