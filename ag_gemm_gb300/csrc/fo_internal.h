// Internal declarations shared by the host-side translation units of
// libflashoverlap.so. Not part of the public ABI (see include/flashoverlap.h).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "flashoverlap.h"

#define FO_MAX_R 16

// Tile shape of the chunk GEMM: one CTA owns a 128 x 256 fp32 accumulator in
// tensor memory; a pipeline stage holds 128 bytes of the reduction dimension
// (64 bf16 or 32 fp32 elements) of both operands.
#define FO_BM 128
#define FO_BN 256
#define FO_BK_BYTES 128

struct fo_transfer { int32_t src, dst, chunk, step; };
struct fo_edge { int32_t ra, sa, rb, sb; };

struct fo_plan_s {
  fo_plan_desc d;
  int R;
  // table[r][s]: chunk (RS/DP: owner of the partial) or source shard (AG)
  // handled by rank r at step s.
  int32_t table[FO_MAX_R][FO_MAX_R];
  // task_r[i], task_s[i]: rank and step of the i-th chunk task in the
  // kernel's order (see fo_interleave). Within one lockstep step the RS/DP
  // ranks alternate direction from step to step, so the shards written last
  // in step s are the first ones written in step s+1.
  int32_t task_r[FO_MAX_R * FO_MAX_R];
  int32_t task_s[FO_MAX_R * FO_MAX_R];
  // ord[r][s]: how many partials of the same chunk come before (r, s) in the
  // kernel's tile order; 0 = the first partial, which stores instead of adds.
  int32_t ord[FO_MAX_R][FO_MAX_R];
  std::vector<fo_transfer> transfers;
  std::vector<fo_edge> edges;

  // Derived sizes of one chunk task.
  int64_t rows_per_chunk;  // M / R: rows of one chunk of the output (RS/DP) or of one shard (AG)
  int64_t k_red;           // reduction length of one task
  int64_t n_out;           // output columns of one task
  int elem_bytes;          // 2 (bf16) or 4 (fp32 -> tf32 MMA)
  bool pair;               // CTA-pair 256 x 256 tiles (else single-CTA 128 x 256)
  int tiles_m, tiles_n, num_kb;   // tiles_m: m-tiles per chunk of the chosen tile height
  int ctr_tiles_m;         // 128-row tiles per chunk in the counter array (covers both heights)
  int pieces;              // AG: 32-row pieces per shard (mover / ready-flag granularity)

  // Workspace layout.
  size_t ws_bytes;
  size_t ws_counters_off;  // RS/DP: uint32 [R][tiles_m*tiles_n][4]
  size_t ws_flags_off;     // AG copy transport: uint32 [R][R][pieces]
  size_t ws_shard_off;     // bf16 output: fp32 shard sums, R x align256(rows/R * N * 4)
  size_t ws_shard_stride;
  size_t ws_ring_off;      // ring RS: rank q's fp32 receive buffer [M x N] at off + q * stride
  size_t ws_ring_stride;
  bool ring;               // d.rs_algo == FO_RS_RING
  size_t ws_wt_off;        // fp32 inputs with W as [K x N]: W_r^T [N x K_r] fp32 at off + r * stride
  size_t ws_wt_stride;
  size_t ws_trace_off;     // trace = 1: uint64 [FO_TRACE_MAX_CTAS][FO_TRACE_STAMPS]
  int32_t last_grid;       // CTAs of the last fused-kernel launch (0 = none yet)
  // Tail split: room for sk_cap split tiles (0 = none reserved): their fp32
  // partials at ws_split_off (sk_cap x tile rows x FO_BN) and their release
  // counters [sk_cap][2][4] at ws_split_ctr_off. The split region ends the
  // workspace; everything else fits in the first ws_split_off bytes.
  int32_t sk_cap;
  size_t ws_split_off, ws_split_ctr_off;
  int32_t last_split_tiles;

  int32_t last_launches;
  void* param_cache;       // host copy of the last kernel parameter block
  int param_cache_kind;    // which call built it (0 = none)
  const void* param_cache_key[4 * FO_MAX_R];  // the pointers it was built from (X/A, W/B, Y/D, G)
  const void* param_cache_ws;                 // and the workspace, where the maps point into it
};

// Workspace header (offset 0): device status word and launch epoch.
struct fo_ws_header {
  int32_t code;            // 0 or FO_ERR_TIMEOUT
  int32_t rank, step, chunk;
  uint32_t epoch;          // incremented by the last CTA of every AG launch
  uint32_t exit_count;     // CTAs of the current AG launch that finished
  uint32_t pad[10];
};

// Helpers of fo_api.cu used by the allocation-free entry point
// (fo_noalloc.cu). FoParams is declared in fo_kernel.cuh.
namespace fo { struct FoParams; }
fo_status fo_internal_check_ptrs(int R, const void* const* a);
fo_status fo_internal_check_device_ptrs(int R, const void* const* a, fo_stream_t stream);
fo_status fo_internal_rs_params_nocache(fo_plan_t p, const void* const* X, const void* const* W,
                                        void* const* Y, void* scratch, fo::FoParams* k, int* variant,
                                        int* grid);

// Host logging (FO_LOG=1 in the environment): plan summaries and launches.
bool fo_log_enabled();

// Units of a GB300 (152 SMs) for a plan's tile shape: 76 CTA pairs or 152
// CTAs. Used to size the tail split's workspace at plan time.
#define FO_GB300_SMS 152

// Tiles to cut along the reduction when `total` tiles run on `units` units:
// the last partial wave plus two whole waves (or every tile, below two
// waves), when the partial wave would leave more than 2% of the launch
// idle; else 0.
int fo_tail_split_tiles(int64_t total, int units);
