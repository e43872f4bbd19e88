// Query-split attention with its row-parallel output projection on sm_103a.
//
// Tensor-parallel attention: rank r holds `heads` heads of dimension 128,
// Q_r, K_r, V_r [T x heads*128] bf16 for every token, and its slice Wo_r of
// the output projection. Query-split attention (gist.science, "Technical
// Summary" section 2, "Architectural Versatility": scores, softmax and the
// weighted sum decomposed so that more compute overlaps the communication)
// splits the queries into R blocks; rank r's step s takes query block
// c = (r - 1 - s) mod R, the Flash-RS order, so the block that stays on the
// rank comes last. Block c's attention output rows are the rows of chunk c
// of the projection's reduce-scatter.
//
// fo_attn_rs runs two launches on one stream:
//   1. fo_attn_kernel: the attention of every (rank, step, head, 128-query
//      tile) in the plan's task order, O_r = softmax(Q K^T / sqrt(128) +
//      mask) V, written bf16 into the caller's O_r;
//   2. the fused GEMM + reduce-scatter (fo_gemm_rs) of O_r . Wo_r.
// On one GPU the reduce-scatter's transfers are the second launch's L2
// reduce-adds, already overlapped with its own math; the first launch
// computes the attention in the same query-block order.
//
// fo_attn_kernel, one CTA per SM, persistent over work items, which CTAs
// take dynamically (the costlier query tiles of a block first, since under
// the causal mask a tile's cost grows with its position):
//   warp 0     TMA producer: the item's Q tile (128 x 128) once, then K and
//              V blocks of 128 keys into two-stage rings, K one block ahead;
//   warp 1     TMEM allocation; MMA issue: S_j = Q K_j^T into one of two
//              TMEM score buffers, then O += P_{j-1} V_{j-1} once the softmax
//              warps have written P_{j-1}, so S_j overlaps softmax(j-1);
//   warps 2-5  softmax, one query row per thread: the row's 128 scores from
//              TMEM, the running maximum and sum (online softmax), P in bf16
//              into shared memory as the next MMA's A operand, and the
//              rescale of the TMEM output row when the maximum grows by more
//              than 8 in log2 units (a smaller growth keeps the old maximum:
//              the weights then stay below 2^8 and the final division by the
//              sum cancels the choice); at the item's end O / sum, bf16, TMA
//              store.
// Every wait is bounded; a wait that runs out raises the CTA's abort flag and
// records FO_ERR_TIMEOUT in the workspace status word.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "fo_device.cuh"
#include "fo_internal.h"

namespace fo_attn {

using namespace fo;

constexpr int kHeadDim = 128;
constexpr int kTile = 128;                       // query rows per item, keys per block
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;   // 32 KB of bf16
constexpr uint32_t kHalf = kTileBytes / 2;              // one 64-column half: 128 rows x 128 B
constexpr int kKStages = 3;   // K blocks in flight (each is free again once its scores are computed)
constexpr int kVStages = 2;   // V blocks in flight (free once their weighted sum is computed)
// Shared memory, from a 1024-byte aligned base: Q, the K and V rings, one P
// buffer (P_j is written once the weighted sum of P_{j-1} has completed),
// barriers.
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kVStages * kTileBytes;
constexpr uint32_t kOffBar = kOffP + kTileBytes;
constexpr int kSmemBytes = 1024 + (int)kOffBar + 512;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleLog2 = 8.0f;

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, A
// K-major, B K-major (scores) or MN-major (weighted sum), M = N = 128.
__host__ __device__ constexpr uint32_t idesc(bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(kTile >> 3) << 17) |
         ((uint32_t)(kTile >> 4) << 24);
}

struct AttnParams {
  CUtensorMap tmQ[FO_MAX_R];   // Q_r [T x heads*128], box 64 x 128
  CUtensorMap tmK[FO_MAX_R];   // K_r, box 64 x 128
  CUtensorMap tmV[FO_MAX_R];   // V_r, box 64 x 64
  CUtensorMap tmO[FO_MAX_R];   // O_r, box 64 x 32 (stores)
  int32_t table[FO_MAX_R][FO_MAX_R];
  int32_t task_r[FO_MAX_R * FO_MAX_R];
  int32_t task_s[FO_MAX_R * FO_MAX_R];
  int32_t R, T, heads, causal, qtiles;   // qtiles: 128-row query tiles per block of T/R rows
  float scale_log2;                      // log2(e) / sqrt(128)
  int32_t* status;
};

struct Item {
  int r, s, c, h, q0, nkb;
};

__device__ __forceinline__ Item decode(const AttnParams& p, int L) {
  const int per_task = p.heads * p.qtiles;
  const int task = L / per_task;
  const int rem = L - task * per_task;
  Item it;
  it.r = p.task_r[task];
  it.s = p.task_s[task];
  it.c = p.table[it.r][it.s];
  it.h = rem / p.qtiles;
  const int qt = p.qtiles - 1 - (rem - it.h * p.qtiles);   // the costlier (later) query tiles first
  it.q0 = it.c * (p.T / p.R) + qt * kTile;
  it.nkb = p.causal ? it.q0 / kTile + 1 : p.T / kTile;
  return it;
}

// Row `row` (one per thread) of a 128-row, 64-column bf16 half in the
// 128B-swizzle layout: 16-byte chunk j of the row sits at chunk j ^ (row % 8).
template <int NW>
__device__ __forceinline__ void store_row_half(uint32_t half_base, int row, const uint32_t (&w)[NW], int w0) {
  const uint32_t rb = half_base + (uint32_t)row * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = rb + ((uint32_t)(j ^ (row & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[w0 + 4 * j]), "r"(w[w0 + 4 * j + 1]),
                 "r"(w[w0 + 4 * j + 2]), "r"(w[w0 + 4 * j + 3])
                 : "memory");
  }
}

// 2^x by the multi-function unit's approximate base-2 exponential
// (PTX ex2.approx.ftz.f32; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// D[tmem] (+)= A[tmem] x B[smem]: the A operand read from tensor memory
// (128 lanes = 128 rows, two 16-bit elements per 32-bit column).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1) fo_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP, sBar = base + kOffBar;
  // Barrier slots (8 bytes each) in the barrier area.
  enum : int {
    kBarQFull = 0, kBarQEmpty, kBarOFree, kBarMmaDone, kBarSlot,   // kBarSlot: TMEM address, abort flag
    kBarPFull = 5,       // two: the softmax warps wrote P_j (and a rescaled O)
    kBarPvDone = 7,      // two: P_j V_j completed
    kBarVFull = 9,       // kVStages
    kBarVEmpty = 11,     // kVStages
    kBarKFull = 13,      // kKStages
    kBarKEmpty = 16,     // kKStages
    kBarSFull = 19,      // three score buffers
    kBarSFree = 22,      // three
    kBarItemFull = 25,   // two item slots
    kBarItemFree = 27,   // two
    kBarItemSlot = 29,   // the two item indices
    kBarCount = 30
  };
  static_assert(kBarCount * 8 <= 512, "barrier area");
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };
  const uint32_t q_full = bar(kBarQFull), q_empty = bar(kBarQEmpty), o_free = bar(kBarOFree);
  auto k_full = [&](int st) { return bar(kBarKFull + st); };
  auto k_empty = [&](int st) { return bar(kBarKEmpty + st); };
  auto v_full = [&](int st) { return bar(kBarVFull + st); };
  auto v_empty = [&](int st) { return bar(kBarVEmpty + st); };
  auto s_full = [&](int b) { return bar(kBarSFull + b); };
  auto s_free = [&](int b) { return bar(kBarSFree + b); };
  auto p_full = [&](int b) { return bar(kBarPFull + b); };
  auto pv_done = [&](int b) { return bar(kBarPvDone + b); };
  const uint32_t sSlot = bar(kBarSlot);
  // Work items are dealt dynamically: the producer takes the next item index
  // from a counter in the workspace header and passes it to the MMA and
  // softmax warps through a two-slot ring.
  auto item_full = [&](int sl) { return bar(kBarItemFull + sl); };
  auto item_free = [&](int sl) { return bar(kBarItemFree + sl); };
  volatile int32_t* item_slot = reinterpret_cast<volatile int32_t*>(gbase + (bar(kBarItemSlot) - base));
  uint32_t* const ctr = reinterpret_cast<uint32_t*>(p.status) + 6;   // header pad words: next item, CTAs done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + (sSlot - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (sSlot - base) + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = p.R * p.R * p.heads * p.qtiles;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 4);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(k_full(i), 1);
      mbar_init(k_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(v_full(i), 1);
      mbar_init(v_empty(i), 1);
      mbar_init(s_full(i), 1);
      mbar_init(s_free(i), 1);
      if (i == 1) {
        mbar_init(s_full(2), 1);
        mbar_init(s_free(2), 1);
      }
      mbar_init(p_full(i), 4);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(bar(kBarMmaDone), 1);   // every MMA issued has completed (before TMEM is freed)
    for (int sl = 0; sl < 2; ++sl) {
      mbar_init(item_full(sl), 1);
      mbar_init(item_free(sl), 5);   // the MMA thread and the four softmax warps
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc<1>(sSlot, 512);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // S buffers at columns 0, 128 and 256, O at 384
  constexpr uint32_t kOCol = 384;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // K blocks run two ahead of V blocks, as the scores do: K_j is free
      // again once S_j is computed, V_j only once P_j V_j is.
      uint32_t gk = 0, gv = 0;   // K and V blocks loaded so far (both number the CTA's blocks)
      int n = 0, nq = 0;         // items taken, Q tiles loaded
      bool ok = true;
      auto load_k = [&](const Item& it, int j) -> bool {
        const int st = (int)(gk % kKStages);
        if (!mbar_wait(k_empty(st), ((gk / kKStages) & 1u) ^ 1u, abort_flag, kWaitNs)) return false;
        const uint32_t sk = sK + (uint32_t)st * kTileBytes;
        mbar_arrive_expect_tx(k_full(st), kTileBytes);
        tma_load_2d(sk, &p.tmK[it.r], k_full(st), it.h * kHeadDim, j * kTile);
        tma_load_2d(sk + kHalf, &p.tmK[it.r], k_full(st), it.h * kHeadDim + 64, j * kTile);
        ++gk;
        return true;
      };
      auto load_v = [&](const Item& it, int j) -> bool {
        const int st = (int)(gv & 1u);
        if (!mbar_wait(v_empty(st), ((gv >> 1) & 1u) ^ 1u, abort_flag, kWaitNs)) return false;
        const uint32_t sv = sV + (uint32_t)st * kTileBytes;
        mbar_arrive_expect_tx(v_full(st), kTileBytes);
        // V as the MN-major B operand: per 64 keys, two 64-column boxes.
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
#pragma unroll
          for (int dh = 0; dh < 2; ++dh)
            tma_load_2d(sv + (uint32_t)kh * kHalf + (uint32_t)dh * (kHalf / 2), &p.tmV[it.r], v_full(st),
                        it.h * kHeadDim + dh * 64, j * kTile + kh * 64);
        ++gv;
        return true;
      };
      for (;; ++n) {
        const int sl = n & 1;
        if (!mbar_wait(item_free(sl), ((uint32_t)(n >> 1) & 1u) ^ 1u, abort_flag, kWaitNs)) break;
        const int L = (int)atomicAdd(ctr, 1u);
        item_slot[sl] = L;
        mbar_arrive(item_full(sl));
        if (L >= total) break;
        const Item it = decode(p, L);
        if (!mbar_wait(q_empty, (uint32_t)(n & 1) ^ 1u, abort_flag, kWaitNs)) break;
        mbar_arrive_expect_tx(q_full, kTileBytes);
        tma_load_2d(sQ, &p.tmQ[it.r], q_full, it.h * kHeadDim, it.q0);
        tma_load_2d(sQ + kHalf, &p.tmQ[it.r], q_full, it.h * kHeadDim + 64, it.q0);
        ++nq;
        if (!load_k(it, 0) || (it.nkb > 1 && !load_k(it, 1))) break;
        for (int j = 0; j < it.nkb; ++j) {
          if ((j + 2 < it.nkb && !load_k(it, j + 2)) || !load_v(it, j)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
      }
      // Loads still in flight land before the CTA may exit.
      volatile int never = 0;
      for (uint32_t k = gk > (uint32_t)kKStages ? gk - kKStages : 0u; k < gk; ++k)
        mbar_wait(k_full((int)(k % kKStages)), (k / kKStages) & 1u, &never, 100000000ull);
      for (uint32_t k = gv > 2u ? gv - 2u : 0u; k < gv; ++k)
        mbar_wait(v_full((int)(k & 1u)), (k >> 1) & 1u, &never, 100000000ull);
      if (nq > 0) mbar_wait(q_full, (uint32_t)((nq - 1) & 1), &never, 100000000ull);
      if (*abort_flag) record_error(p.status, FO_ERR_TIMEOUT, -1, -1, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0;
      int n = 0;
      bool ok = true;
      auto pv = [&](uint32_t gp, bool first) -> bool {
        const int b = (int)(gp & 1u);
        if (!mbar_wait(p_full(b), (gp >> 1) & 1u, abort_flag, kWaitNs) ||
            !mbar_wait(v_full(b), (gp >> 1) & 1u, abort_flag, kWaitNs))
          return false;
        if (first && !mbar_wait(o_free, (uint32_t)(n & 1) ^ 1u, abort_flag, kWaitNs)) return false;
        tc_fence_after();
        // A = P_j from TMEM: the first 64 columns of its score buffer, row i
        // in lane i, two bf16 weights per column; 8 columns per 16 keys.
        const uint32_t pa = tmem + (gp % 3u) * 128u;
        const uint32_t vb = sV + (uint32_t)b * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kh = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
          const uint64_t bd = smem_desc_sw128(vb + kh * kHalf + kk * 2048u, kHalf / 2, 1024);
          tc_mma_ts(tmem + kOCol, pa + (uint32_t)k * 8u, bd, idesc(true), (!first || k > 0) ? 1u : 0u);
        }
        tc_commit<1>(pv_done(b));
        tc_commit<1>(v_empty(b));
        tc_commit<1>(s_free(gp % 3u));   // P_j read: the buffer may take scores again
        return true;
      };
      // S_{j+1} is issued before P_j V_j, so a score block waits in the pipe
      // while the softmax warps work on block j. Its buffer last held P_{j-2},
      // whose weighted sum completed before P_{j-1} could be written.
      auto issue_s = [&](uint32_t gs) -> bool {
        const int sb = (int)(gs % 3u);   // score buffer and K stage
        const uint32_t ph = (gs / 3u) & 1u;
        if (!mbar_wait(k_full(sb), ph, abort_flag, kWaitNs) || !mbar_wait(s_free(sb), ph ^ 1u, abort_flag, kWaitNs))
          return false;
        tc_fence_after();
        const uint32_t kb = sK + (uint32_t)sb * kTileBytes;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t kh = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
          const uint64_t ad = smem_desc_sw128(sQ + kh * kHalf + kk * 32u, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + kh * kHalf + kk * 32u, 16, 1024);
          tc_mma<1, false>(tmem + (uint32_t)sb * 128u, ad, bd, idesc(false), k > 0 ? 1u : 0u);
        }
        tc_commit<1>(s_full(sb));
        tc_commit<1>(k_empty(sb));
        return true;
      };
      for (; ok; ++n) {
        const int sl = n & 1;
        if (!mbar_wait(item_full(sl), (uint32_t)(n >> 1) & 1u, abort_flag, kWaitNs)) break;
        const int L = item_slot[sl];
        mbar_arrive(item_free(sl));
        if (L >= total) break;
        const Item it = decode(p, L);
        if (!mbar_wait(q_full, (uint32_t)(n & 1), abort_flag, kWaitNs)) break;
        tc_fence_after();
        const uint32_t g0 = g;
        ok = issue_s(g0);
        if (ok && it.nkb == 1) tc_commit<1>(q_empty);   // every score block of the item issued
        for (int j = 0; j < it.nkb && ok; ++j) {
          if (j + 1 < it.nkb) {
            ok = issue_s(g0 + (uint32_t)j + 1u);
            if (ok && j + 2 == it.nkb) tc_commit<1>(q_empty);
          }
          if (ok) ok = pv(g0 + (uint32_t)j, j == 0);
        }
        g = g0 + (uint32_t)it.nkb;
      }
      // Every issued MMA completes before TMEM is released.
      tc_commit<1>(bar(kBarMmaDone));
      volatile int never = 0;
      mbar_wait(bar(kBarMmaDone), 0, &never, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int row = q * 32 + lane;          // query row within the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t g = 0;
    int n = 0;
    for (;; ++n) {
      const int sl = n & 1;
      if (!mbar_wait(item_full(sl), (uint32_t)(n >> 1) & 1u, abort_flag, kWaitNs)) break;
      const int L = item_slot[sl];
      __syncwarp();
      if (lane == 0) mbar_arrive(item_free(sl));
      if (L >= total) break;
      const Item it = decode(p, L);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < it.nkb; ++j, ++g) {
        const int b = (int)(g & 1u);      // P / weighted-sum barriers
        const int sb = (int)(g % 3u);     // score buffer
        if (!mbar_wait(s_full(sb), (g / 3u) & 1u, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // The row's 128 scores: four TMEM loads, one wait.
        uint32_t v[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_off + (uint32_t)sb * 128u + (uint32_t)cc * 32u, v[cc]);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) reg_fence(v[cc]);
        if (p.causal && j == it.nkb - 1) {
          // The block holding this tile's own keys: key t of the block is
          // query t of the tile, so the row sees keys 0..row.
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (cc * 32 + t > row) v[cc][t] = __float_as_uint(-INFINITY);
        }
        // Maximum and (below) sum over eight independent partial chains: one
        // warp per scheduler has nothing else to hide a serial chain's latency.
        float mxs[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mxs[a] = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int t = 0; t < 32; ++t) mxs[t & 7] = fmaxf(mxs[t & 7], __uint_as_float(v[cc][t]));
        float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                         fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
        mx *= p.scale_log2;   // log2 units (the scale is positive, so the maximum commutes)
        const float m_use = (j == 0 || mx > m + kRescaleLog2) ? fmaxf(m, mx) : m;
        const float alpha = j == 0 ? 0.f : ex2_approx(m - m_use);
        float sums[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) sums[a] = 0.f;
        const float scl = p.scale_log2, neg = -m_use;
        uint32_t w[2][32];
#pragma unroll
        for (int t = 0; t < 64; ++t) {
          const int c0 = 2 * t;
          const float e0 = ex2_approx(fmaf(__uint_as_float(v[c0 >> 5][c0 & 31]), scl, neg));
          const float e1 = ex2_approx(fmaf(__uint_as_float(v[(c0 + 1) >> 5][(c0 + 1) & 31]), scl, neg));
          sums[t & 7] += e0 + e1;
          w[t >> 5][t & 31] = pack_bf16(e0, e1);
        }
        const float sum = ((sums[0] + sums[1]) + (sums[2] + sums[3])) + ((sums[4] + sums[5]) + (sums[6] + sums[7]));
        // P_j in bf16 over the first 64 columns of its own score buffer
        // (the scores are in registers now), the A operand of P_j V_j.
        tmem_st32(tmem + lane_off + (uint32_t)sb * 128u, w[0]);
        tmem_st32(tmem + lane_off + (uint32_t)sb * 128u + 32u, w[1]);
        l = l * alpha + sum;
        m = m_use;
        // Rescale this row of O when its maximum moved (after the weighted
        // sum of the previous block has completed).
        const bool need = j > 0 && alpha < 1.f;
        if (__any_sync(0xffffffffu, need)) {
          const uint32_t gq = g - 1u;
          if (!mbar_wait(pv_done((int)(gq & 1u)), (gq >> 1) & 1u, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float a = need ? alpha : 1.f;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kOCol + (uint32_t)cc * 32u, v);
            tmem_ld_wait();
            reg_fence(v);
#pragma unroll
            for (int t = 0; t < 32; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) * a);
            tmem_st32(tmem + lane_off + kOCol + (uint32_t)cc * 32u, v);
          }
        }
        tmem_st_wait();   // P (and a rescaled O) are in TMEM before the weighted sum may read them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(b));
      }
      if (!ok) break;
      // The item's output: O / l in bf16, staged in this warp's own rows of
      // the P buffer the last weighted sum read (the rows this warp alone
      // writes), then TMA-stored, 64 columns x 32 rows per op.
      const uint32_t gl = g - 1u;
      if (!mbar_wait(pv_done((int)(gl & 1u)), (gl >> 1) & 1u, abort_flag, kWaitNs)) break;
      tc_fence_after();
      if (lane == 0) bulk_wait_read<0>();   // the previous item's output store has read the staging rows
      __syncwarp();
      const float inv = 1.f / l;
      const uint32_t stage = sP + (uint32_t)q * 4096u;
#pragma unroll
      for (int dh = 0; dh < 2; ++dh) {
        uint32_t w[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kOCol + (uint32_t)(dh * 64 + cc * 32), v);
          tmem_ld_wait();
          reg_fence(v);
#pragma unroll
          for (int t = 0; t < 16; ++t)
            w[cc * 16 + t] = pack_bf16(__uint_as_float(v[2 * t]) * inv, __uint_as_float(v[2 * t + 1]) * inv);
        }
        // 32 rows x 128 B per box, rows indexed by lane: the half dh of the
        // P buffer, this warp's 32 rows.
        const uint32_t rb = stage + (uint32_t)dh * kHalf + (uint32_t)lane * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rb + ((uint32_t)(j ^ (lane & 7)) << 4)),
                       "r"(w[4 * j]), "r"(w[4 * j + 1]), "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                       : "memory");
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(o_free);
        tma_store_2d(&p.tmO[it.r], stage, it.h * kHeadDim, it.q0 + q * 32);
        tma_store_2d(&p.tmO[it.r], stage + kHalf, it.h * kHeadDim + 64, it.q0 + q * 32);
        bulk_commit();
      }
      __syncwarp();
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc<1>(tmem, 512);
  }
  // The last CTA to finish resets the item counter for the next launch
  // (every CTA has stopped taking items by then).
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
      atomicExch(ctr, 0u);
      atomicExch(ctr + 1, 0u);
      __threadfence();
    }
  }
}

}  // namespace fo_attn

namespace {

bool enc(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_c, uint32_t box_r) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_c, box_r};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// Checks the arguments of the attention launch and launches it.
fo_status launch_attention(fo_plan_t p, const void* const* Q, const void* const* K, const void* const* V,
                           void* const* O, int32_t heads, int32_t causal, void* ws, fo_stream_t stream) {
  if (!p || !ws) return FO_ERR_INVALID_ARG;
  if (p->d.op != FO_OP_GEMM_RS || p->elem_bytes != 2) return FO_ERR_INVALID_ARG;
  if (heads < 1 || (causal != 0 && causal != 1)) return FO_ERR_INVALID_ARG;
  const int R = p->R;
  const int64_t T = p->d.M, width = (int64_t)heads * fo_attn::kHeadDim;
  if (p->k_red != width) return FO_ERR_SHAPE;            // the projection reads heads * 128 columns per rank
  if ((T / R) % fo_attn::kTile) return FO_ERR_SHAPE;      // whole 128-row query tiles per block
  fo_status st;
  if ((st = fo_internal_check_ptrs(R, Q)) || (st = fo_internal_check_ptrs(R, K)) ||
      (st = fo_internal_check_ptrs(R, V)) || (st = fo_internal_check_ptrs(R, (const void* const*)O)))
    return st;
  if ((st = fo_internal_check_device_ptrs(R, Q, stream)) || (st = fo_internal_check_device_ptrs(R, K, stream)) ||
      (st = fo_internal_check_device_ptrs(R, V, stream)) ||
      (st = fo_internal_check_device_ptrs(R, (const void* const*)O, stream)))
    return st;
  int dev = 0, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return FO_ERR_UNSUPPORTED;
  static_assert(sizeof(fo_attn::AttnParams) <= 32764, "kernel parameters");
  fo_attn::AttnParams k;
  memset(static_cast<void*>(&k), 0, sizeof(k));
  bool ok = true;
  for (int r = 0; r < R && ok; ++r) {
    ok &= enc(&k.tmQ[r], Q[r], (uint64_t)width, (uint64_t)T, 64, 128);
    ok &= enc(&k.tmK[r], K[r], (uint64_t)width, (uint64_t)T, 64, 128);
    ok &= enc(&k.tmV[r], V[r], (uint64_t)width, (uint64_t)T, 64, 64);
    ok &= enc(&k.tmO[r], O[r], (uint64_t)width, (uint64_t)T, 64, 32);
  }
  if (!ok) return FO_ERR_CUDA;
  memcpy(k.table, p->table, sizeof(k.table));
  memcpy(k.task_r, p->task_r, sizeof(k.task_r));
  memcpy(k.task_s, p->task_s, sizeof(k.task_s));
  k.R = R;
  k.T = (int32_t)T;
  k.heads = heads;
  k.causal = causal;
  k.qtiles = (int32_t)(T / R / fo_attn::kTile);
  k.scale_log2 = (float)(1.4426950408889634 / sqrt((double)fo_attn::kHeadDim));
  k.status = static_cast<int32_t*>(ws);
  const int total = R * R * heads * k.qtiles;
  const int grid = total < sms ? total : sms;
  auto kern = fo_attn::fo_attn_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fo_attn::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return FO_ERR_CUDA;
  }
  kern<<<grid, fo_attn::kThreads, fo_attn::kSmemBytes, (cudaStream_t)stream>>>(k);
  const cudaError_t e = cudaGetLastError();
  if (fo_log_enabled())
    fprintf(stderr, "[flashoverlap] attention R=%d T=%lld heads=%d causal=%d: %d items on %d CTAs: %s\n", R,
            (long long)T, heads, causal, total, grid, cudaGetErrorString(e));
  if (e != cudaSuccess) return FO_ERR_CUDA;
  p->last_launches = 1;
  return FO_OK;
}

}  // namespace

extern "C" fo_status fo_attention(fo_plan_t p, const void* const* Q, const void* const* K, const void* const* V,
                                  void* const* O, int32_t heads, int32_t causal, void* ws, fo_stream_t stream) {
  return launch_attention(p, Q, K, V, O, heads, causal, ws, stream);
}

extern "C" fo_status fo_attn_rs(fo_plan_t p, const void* const* Q, const void* const* K, const void* const* V,
                                const void* const* Wo, void* const* O, void* const* Y, int32_t heads,
                                int32_t causal, void* ws, fo_stream_t stream) {
  fo_status st;
  if (p && ((st = fo_internal_check_ptrs(p->R, Wo)) || (st = fo_internal_check_ptrs(p->R, (const void* const*)Y))))
    return st;
  if ((st = launch_attention(p, Q, K, V, O, heads, causal, ws, stream))) return st;
  // The projection's fused GEMM + reduce-scatter of O_r . Wo_r.
  if ((st = fo_gemm_rs(p, (const void* const*)O, Wo, Y, ws, stream))) return st;
  p->last_launches = 2;
  return FO_OK;
}
