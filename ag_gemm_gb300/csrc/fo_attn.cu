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
// fo_attention runs the first launch alone. On one GPU the reduce-scatter's transfers are the second launch's L2
// reduce-adds, already overlapped with its own math; the first launch
// computes the attention in the same query-block order.
//
// fo_attn_kernel, one CTA per SM, persistent over work items (one item =
// one rank, step, head and 128-query tile), which CTAs take one at a time
// from a counter in the workspace header, the costlier query tiles of a
// block first (under the causal mask a tile's cost grows with its
// position):
//   warp 0      TMA producer: the item's Q tile (128 x 128) once, then K
//               blocks of 128 keys into a three-stage ring and V blocks into
//               a two-stage ring, K two blocks ahead of V;
//   warp 1      TMEM allocation; S_j = Q K_j^T into score buffer j mod 3
//               (of three), up to two blocks ahead of the softmax;
//   warp 2      O += P_j V_j, with P_j read from TMEM (the "A in tensor
//               memory" form), once the softmax warps have written it. The
//               two MMA streams come from two warps because a thread that
//               issues tcgen05.mma runs only a few instructions ahead of the
//               tensor pipe: one issuer would hold the score MMAs back while
//               it waits for the softmax;
//   warps 3-10  softmax: two warps per 32-row quarter of the tile, each over
//               64 of a block's 128 keys. A thread takes its row's 64 scores
//               from TMEM, the two warps swap partial row maxima (each
//               computes its weights with the running maximum while the
//               partner's value is in flight, and again only if the
//               maximum moved), and each writes its bf16 weights over its
//               own score columns. The
//               running maximum only moves when it grows by more than 8 in
//               log2 units (a smaller growth keeps the old one: the weights
//               then stay below 2^8 and the final division by the sum
//               cancels the choice); when it moves, each warp rescales its 64
//               columns of the TMEM output row. At the item's end the partial
//               sums are swapped and O / sum is stored in bf16 from registers.
// Every wait gives up after 2 s; a wait that runs out raises the CTA's abort
// flag, every role leaves its loops, and the CTA records FO_ERR_TIMEOUT in
// the workspace status word.
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
// Warps: 0 TMA producer, 1 score MMAs (and TMEM allocation), 2 weighted-sum
// MMAs, 3-10 softmax.
constexpr int kThreads = 352;
constexpr int kSoftWarp0 = 3;
// Registers are capped as for 384 threads (168 a thread): three of the
// eleven warps share each of schedulers 0-2, and a scheduler's register file
// holds three warps of at most 170 registers.
constexpr int kRegBoundThreads = 384;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;   // 32 KB of bf16
constexpr uint32_t kHalf = kTileBytes / 2;              // one 64-column half: 128 rows x 128 B
constexpr int kKStages = 3;   // K blocks in flight (each is free again once its scores are computed)
constexpr int kVStages = 2;   // V blocks in flight (free once their weighted sum is computed)
// Shared memory, from a 1024-byte aligned base: Q, the K and V rings, the
// softmax warps' mailboxes (8 warps x 2 parities x 32 lanes x 8 bytes),
// barriers.
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffX = kOffV + kVStages * kTileBytes;
constexpr uint32_t kMailboxWords = 8 * 2 * 32;
constexpr uint32_t kOffBar = kOffX + kMailboxWords * 8;
constexpr int kSmemBytes = 1024 + (int)kOffBar + 512;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint64_t kWaitNs = 2000000000ull;   // every wait's bound
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
  uint16_t* O[FO_MAX_R];       // O_r [T x heads*128] bf16, row stride ld elements
  int32_t table[FO_MAX_R][FO_MAX_R];
  int32_t task_r[FO_MAX_R * FO_MAX_R];
  int32_t task_s[FO_MAX_R * FO_MAX_R];
  int32_t R, T, heads, causal, qtiles;   // qtiles: 128-row query tiles per block of T/R rows
  int32_t ld;                            // heads * 128
  float scale_log2;                      // log2(e) / sqrt(128)
  int32_t* status;
  // Test hook (the plan's FO_INJECT_SKIP_SIGNAL): the first softmax warp of
  // CTA 0 does not report its first weights, so that CTA's weighted-sum
  // wait runs out and the launch reports FO_ERR_TIMEOUT.
  int32_t skip_signal;
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

// Packed fp32 pairs (PTX .f32x2 arithmetic, sm_100 and later): each lane of
// the pair is rounded exactly as the scalar instruction would round it.
using f32x2 = unsigned long long;
__device__ __forceinline__ f32x2 f2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(f32x2 r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// Maximum of three (one instruction).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__global__ void __launch_bounds__(kRegBoundThreads, 1) fo_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sBar = base + kOffBar;
  // Barrier slots (8 bytes each). Per-block barriers have three slots,
  // indexed by the block's number mod 3, so that a slot's next phase always
  // depends on the waiter's own progress and a parity wait is never
  // ambiguous.
  enum : int {
    kBarQFull = 0, kBarQEmpty, kBarOFree, kBarSlot,   // kBarSlot: TMEM address, abort flag
    kBarSDone, kBarPvDoneAll,                         // every score / weighted-sum MMA issued has completed
    kBarKFull = 6,      // kKStages: K block loaded
    kBarVFull = 9,      // kVStages: V block loaded
    kBarSFull = 11,     // 3: S_j computed (also: K stage j mod 3 free again)
    kBarPFull = 14,     // 3: the softmax warps wrote P_j (and a rescaled O)
    kBarPvDone = 17,    // 3: P_j V_j computed (also: V stage free, score buffer free)
    kBarItemFull = 20,  // 2 item slots
    kBarItemFree = 22,  // 2
    kBarItemSlot = 24,  // the two item indices
    kBarCount = 25
  };
  static_assert(kBarCount * 8 <= 512, "barrier area");
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };
  const uint32_t q_full = bar(kBarQFull), q_empty = bar(kBarQEmpty), o_free = bar(kBarOFree);
  auto k_full = [&](uint32_t gk) { return bar(kBarKFull + (int)(gk % 3u)); };
  auto v_full = [&](uint32_t gv) { return bar(kBarVFull + (int)(gv & 1u)); };
  auto s_full = [&](uint32_t g) { return bar(kBarSFull + (int)(g % 3u)); };
  auto p_full = [&](uint32_t g) { return bar(kBarPFull + (int)(g % 3u)); };
  auto pv_done = [&](uint32_t g) { return bar(kBarPvDone + (int)(g % 3u)); };
  // Parity of block g's phase on its mod-3 slot.
  auto ph3 = [](uint32_t g) { return (g / 3u) & 1u; };
  const uint32_t sSlot = bar(kBarSlot);
  // Work items are dealt dynamically: the producer takes the next item index
  // from a counter in the workspace header and passes it to the other warps
  // through a two-slot ring.
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
    mbar_init(o_free, 8);   // every softmax warp has read its O columns
    mbar_init(bar(kBarSDone), 1);
    mbar_init(bar(kBarPvDoneAll), 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarPFull + i), 8);
      mbar_init(bar(kBarPvDone + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(item_full(i), 1);
      mbar_init(item_free(i), 10);   // both MMA issuers and the eight softmax warps
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  {
    volatile unsigned long long* mb = reinterpret_cast<volatile unsigned long long*>(gbase + kOffX);
    for (uint32_t i = threadIdx.x; i < kMailboxWords; i += kThreads) mb[i] = 0ull;
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

  // Takes item n from its ring slot (every consumer role, one arrival each).
  auto take_item = [&](int n, int& L) -> bool {
    const int sl = n & 1;
    if (!mbar_wait(item_full(sl), (uint32_t)(n >> 1) & 1u, abort_flag, kWaitNs)) return false;
    L = item_slot[sl];
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // K blocks run two ahead of V blocks: K_j's stage is free again once
      // S_j is computed, V_j's once P_j V_j is.
      uint32_t gk = 0, gv = 0;   // K and V blocks loaded so far (both number the CTA's blocks)
      int n = 0, nq = 0;         // items taken, Q tiles loaded
      bool ok = true;
      auto load_k = [&](const Item& it, int j) -> bool {
        if (gk >= 3u && !mbar_wait(s_full(gk - 3u), ph3(gk - 3u), abort_flag, kWaitNs)) return false;
        const uint32_t sk = sK + (gk % 3u) * kTileBytes;
        mbar_arrive_expect_tx(k_full(gk), kTileBytes);
        tma_load_2d(sk, &p.tmK[it.r], k_full(gk), it.h * kHeadDim, j * kTile);
        tma_load_2d(sk + kHalf, &p.tmK[it.r], k_full(gk), it.h * kHeadDim + 64, j * kTile);
        ++gk;
        return true;
      };
      auto load_v = [&](const Item& it, int j) -> bool {
        if (gv >= 2u && !mbar_wait(pv_done(gv - 2u), ph3(gv - 2u), abort_flag, kWaitNs)) return false;
        const uint32_t sv = sV + (gv & 1u) * kTileBytes;
        mbar_arrive_expect_tx(v_full(gv), kTileBytes);
        // V as the MN-major B operand: per 64 keys, two 64-column boxes.
#pragma unroll
        for (int kh = 0; kh < 2; ++kh)
#pragma unroll
          for (int dh = 0; dh < 2; ++dh)
            tma_load_2d(sv + (uint32_t)kh * kHalf + (uint32_t)dh * (kHalf / 2), &p.tmV[it.r], v_full(gv),
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
      for (uint32_t k = gk > 3u ? gk - 3u : 0u; k < gk; ++k) mbar_wait(k_full(k), ph3(k), &never, 100000000ull);
      for (uint32_t k = gv > 2u ? gv - 2u : 0u; k < gv; ++k)
        mbar_wait(v_full(k), (k >> 1) & 1u, &never, 100000000ull);
      if (nq > 0) mbar_wait(q_full, (uint32_t)((nq - 1) & 1), &never, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ score MMAs
    // S_j = Q K_j^T into score buffer j mod 3, as soon as K_j has landed and
    // the weighted sum of P_{j-3} (the buffer's previous contents) is done:
    // up to two blocks ahead of the softmax. A thread that issues
    // tcgen05.mma runs at most a few instructions ahead of the tensor pipe,
    // so the score and weighted-sum streams come from two warps: neither
    // stream's waits hold up the other.
    if (lane == 0) {
      uint32_t g = 0;
      int n = 0;
      for (;; ++n) {
        int L;
        if (!take_item(n, L)) break;
        mbar_arrive(item_free(n & 1));
        if (L >= total) break;
        const Item it = decode(p, L);
        if (!mbar_wait(q_full, (uint32_t)(n & 1), abort_flag, kWaitNs)) break;
        bool ok = true;
        for (int j = 0; j < it.nkb; ++j, ++g) {
          if (!mbar_wait(k_full(g), ph3(g), abort_flag, kWaitNs) ||
              (g >= 3u && !mbar_wait(pv_done(g - 3u), ph3(g - 3u), abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sb = g % 3u;
          const uint32_t kb = sK + sb * kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t kh = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
            const uint64_t ad = smem_desc_sw128(sQ + kh * kHalf + kk * 32u, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kb + kh * kHalf + kk * 32u, 16, 1024);
            tc_mma<1, false>(tmem + sb * 128u, ad, bd, idesc(false), k > 0 ? 1u : 0u);
          }
          tc_commit<1>(s_full(g));
        }
        if (!ok) break;
        tc_commit<1>(q_empty);   // every score block of the item issued
      }
      // Every issued MMA completes before TMEM is released.
      tc_commit<1>(bar(kBarSDone));
      volatile int never = 0;
      mbar_wait(bar(kBarSDone), 0, &never, 100000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ weighted-sum MMAs
    if (lane == 0) {
      uint32_t g = 0;
      int n = 0;
      for (;; ++n) {
        int L;
        if (!take_item(n, L)) break;
        mbar_arrive(item_free(n & 1));
        if (L >= total) break;
        const Item it = decode(p, L);
        bool ok = true;
        for (int j = 0; j < it.nkb; ++j, ++g) {
          if (!mbar_wait(p_full(g), ph3(g), abort_flag, kWaitNs) ||
              !mbar_wait(v_full(g), (g >> 1) & 1u, abort_flag, kWaitNs) ||
              (j == 0 && !mbar_wait(o_free, (uint32_t)(n & 1) ^ 1u, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A = P_j from TMEM, in its score buffer: row i in lane i, two
          // bf16 weights per column, 8 columns per 16 keys; keys 0-63 in
          // columns 0-31, keys 64-127 in columns 64-95 (each softmax warp
          // writes its weights over the first half of its own 64 score
          // columns).
          const uint32_t pa = tmem + (g % 3u) * 128u;
          const uint32_t vb = sV + (g & 1u) * kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t kh = (uint32_t)(k >> 2), kk = (uint32_t)(k & 3);
            const uint64_t bd = smem_desc_sw128(vb + kh * kHalf + kk * 2048u, kHalf / 2, 1024);
            tc_mma_ts(tmem + kOCol, pa + kh * 64u + kk * 8u, bd, idesc(true), (j > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit<1>(pv_done(g));
        }
        if (!ok) break;
      }
      tc_commit<1>(bar(kBarPvDoneAll));
      volatile int never = 0;
      mbar_wait(bar(kBarPvDoneAll), 0, &never, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31, its quarter of
    // the query rows. Warps 3-6 take keys 0-63 of every block and columns
    // 0-63 of O, warps 7-10 keys 64-127 and columns 64-127. The two warps of
    // a quarter swap their partial row maxima every block, and their partial
    // row sums at the item's end, through mailboxes in shared memory: one
    // 64-bit word per lane holds the exchange's sequence number and value,
    // and the reader waits (bounded) for the number it expects.
    const int q = warp & 3;                 // TMEM lane quarter of this warp
    const int sw = warp - kSoftWarp0;       // softmax warp 0..7
    const int half = sw >> 2;               // which 64 keys / O columns
    const int row = q * 32 + lane;          // query row within the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    volatile unsigned long long* const mbox = reinterpret_cast<volatile unsigned long long*>(gbase + kOffX);
    uint32_t x = 0;                         // exchanges so far
    const bool skip_first = p.skip_signal != 0 && blockIdx.x == 0 && sw == 0;   // test hook
    // Two mailboxes a lane, by the exchange's parity: exchange x + 2
    // overwrites exchange x's word only after this warp has read the
    // partner's x + 1, which the partner writes after reading x.
    auto post = [&](float mine) {
      ++x;
      mbox[(sw * 2 + (int)(x & 1u)) * 32 + lane] = ((unsigned long long)x << 32) | __float_as_uint(mine);
    };
    auto fetch = [&](float& theirs) -> bool {
      volatile unsigned long long* const t = mbox + (((sw ^ 4) * 2 + (int)(x & 1u)) * 32 + lane);
      unsigned long long w = *t;
      if ((uint32_t)(w >> 32) != x) {
        const uint64_t t0 = globaltimer();
        uint32_t n = 0;
        while ((uint32_t)((w = *t) >> 32) != x) {
          if ((++n & 63u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) {
              *abort_flag = 1;
              return false;
            }
          }
        }
      }
      theirs = __uint_as_float((uint32_t)w);
      return true;
    };
    uint32_t g = 0;
    for (int n = 0;; ++n) {
      int L;
      if (!take_item(n, L)) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(item_free(n & 1));
      if (L >= total) break;
      const Item it = decode(p, L);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int j = 0; j < it.nkb; ++j, ++g) {
        if (!mbar_wait(s_full(g), ph3(g), abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // This warp's 64 scores of the row: two TMEM loads, one wait.
        const uint32_t scol = tmem + lane_off + (g % 3u) * 128u + (uint32_t)half * 64u;
        uint32_t v[2][32];
        tmem_ld32(scol, v[0]);
        tmem_ld32(scol + 32u, v[1]);
        tmem_ld_wait();
        reg_fence(v[0]);
        reg_fence(v[1]);
        if (p.causal && j == it.nkb - 1) {
          // The block holding this tile's own keys: key t of the block is
          // query t of the tile, so the row sees keys 0..row.
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (half * 64 + cc * 32 + t > row) v[cc][t] = __float_as_uint(-INFINITY);
        }
        // This half's row maximum (raw scores): three-input maxima over eight
        // independent chains.
        float mxs[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mxs[a] = -INFINITY;
#pragma unroll
        for (int t = 0; t < 32; ++t)
          mxs[t & 7] = max3(mxs[t & 7], __uint_as_float(v[t >> 4][(2 * t) & 31]),
                            __uint_as_float(v[t >> 4][(2 * t + 1) & 31]));
        const float mxl = max3(max3(mxs[0], mxs[1], mxs[2]), max3(mxs[3], mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])) *
                          p.scale_log2;   // log2 units (the scale is positive)
        post(mxl);
        // 2^(s * scale - m) for the row's 64 keys: the argument by packed
        // FMAs, the power on the MUFU, the row sum over four packed chains,
        // the weights packed to bf16.
        float sum = 0.f;
        uint32_t w[32];
        auto exps = [&](float mm) {
          const f32x2 scl2 = f2(p.scale_log2, p.scale_log2), neg2 = f2(-mm, -mm);
          f32x2 acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            float x0, x1;
            f2_split(fma2(f2(__uint_as_float(v[t >> 4][(2 * t) & 31]), __uint_as_float(v[t >> 4][(2 * t + 1) & 31])),
                          scl2, neg2),
                     x0, x1);
            const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
            acc[t & 3] = add2(acc[t & 3], f2(e0, e1));
            w[t] = pack_bf16(e0, e1);
          }
          float s0, s1, s2, s3;
          f2_split(add2(acc[0], acc[1]), s0, s1);
          f2_split(add2(acc[2], acc[3]), s2, s3);
          sum = (s0 + s1) + (s2 + s3);
        };
        // While the partner's maximum is on its way, compute the weights with
        // the running maximum: they are final unless the maximum moves (by
        // more than 8), which a half whose own maximum stays below m + 8
        // learns from the partner's value. Weights computed this way are at
        // most 2^8.
        const bool spec = j > 0 && mxl <= m + kRescaleLog2;
        if (spec) exps(m);
        float mx_other;
        if (!__all_sync(0xffffffffu, fetch(mx_other))) {
          ok = false;
          break;
        }
        const float mx = fmaxf(mxl, mx_other);
        const float m_use = (j == 0 || mx > m + kRescaleLog2) ? fmaxf(m, mx) : m;
        const float alpha = j == 0 ? 0.f : ex2_approx(m - m_use);
        if (!spec || m_use != m) exps(m_use);
        // P_j in bf16 over the first 32 of this warp's score columns (the
        // scores are in registers now), the A operand of P_j V_j.
        tmem_st32(scol, w);
        l = l * alpha + sum;
        m = m_use;
        // Rescale this warp's half of the O row when the maximum moved
        // (after the weighted sum of the previous block has completed).
        const bool need = j > 0 && alpha < 1.f;
        if (__any_sync(0xffffffffu, need)) {
          if (!mbar_wait(pv_done(g - 1u), ph3(g - 1u), abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float a = need ? alpha : 1.f;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const uint32_t oc = tmem + lane_off + kOCol + (uint32_t)(half * 64 + cc * 32);
            uint32_t o[32];
            tmem_ld32(oc, o);
            tmem_ld_wait();
            reg_fence(o);
            const f32x2 a2 = f2(a, a);
#pragma unroll
            for (int t = 0; t < 32; t += 2) {
              float r0, r1;
              f2_split(mul2(f2(__uint_as_float(o[t]), __uint_as_float(o[t + 1])), a2), r0, r1);
              o[t] = __float_as_uint(r0);
              o[t + 1] = __float_as_uint(r1);
            }
            tmem_st32(oc, o);
          }
        }
        tmem_st_wait();   // P (and a rescaled O) are in TMEM before the weighted sum may read them
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !(skip_first && g == 0)) mbar_arrive(p_full(g));
      }
      if (!ok) break;
      // The row's sum over all 128 keys of every block, then the item's
      // output: this warp's 64 columns of O / sum in bf16, stored straight
      // from registers (128 contiguous bytes a row).
      float l_other;
      post(l);
      if (!__all_sync(0xffffffffu, fetch(l_other))) break;
      const float inv = 1.f / (l + l_other);
      if (!mbar_wait(pv_done(g - 1u), ph3(g - 1u), abort_flag, kWaitNs)) break;
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32(tmem + lane_off + kOCol + (uint32_t)half * 64u, o[0]);
      tmem_ld32(tmem + lane_off + kOCol + (uint32_t)half * 64u + 32u, o[1]);
      tmem_ld_wait();
      reg_fence(o[0]);
      reg_fence(o[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);   // the next item's first weighted sum may overwrite O
      uint4* dst = reinterpret_cast<uint4*>(p.O[it.r] + (size_t)(it.q0 + row) * (size_t)p.ld +
                                            (size_t)(it.h * kHeadDim + half * 64));
      const f32x2 inv2 = f2(inv, inv);
      auto scaled = [&](uint32_t a, uint32_t b) {
        float r0, r1;
        f2_split(mul2(f2(__uint_as_float(a), __uint_as_float(b)), inv2), r0, r1);
        return pack_bf16(r0, r1);
      };
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t* s8 = &o[c >> 2][(c & 3) * 8];
        dst[c] = make_uint4(scaled(s8[0], s8[1]), scaled(s8[2], s8[3]), scaled(s8[4], s8[5]), scaled(s8[6], s8[7]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc<1>(tmem, 512);
  }
  // A wait that ran out anywhere in the CTA (every role has left its loops
  // by now) is reported in the workspace status word. The last CTA to
  // finish resets the item counter for the next launch (every CTA has
  // stopped taking items by then).
  if (threadIdx.x == 0) {
    if (*abort_flag) record_error(p.status, FO_ERR_TIMEOUT, -1, -1, 0);
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
    k.O[r] = static_cast<uint16_t*>(O[r]);
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
  k.ld = (int32_t)width;
  k.scale_log2 = (float)(1.4426950408889634 / sqrt((double)fo_attn::kHeadDim));
  k.status = static_cast<int32_t*>(ws);
  k.skip_signal = p->d.fault_inject == FO_INJECT_SKIP_SIGNAL ? 1 : 0;
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
