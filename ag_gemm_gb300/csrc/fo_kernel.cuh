// The persistent chunk-GEMM kernel of FlashOverlap on sm_103a.
//
// Every rank's chunk tasks run in that rank's schedule order, the
// rank-adaptive order of Flash-RS / Flash-AG (gist.science, "Technical
// Summary" section 2): for reduce-scatter each rank's own chunk is its last
// task, for all-gather its first. How the R ranks' sequences interleave on
// the one GPU (lockstep, skewed, skewed in slot pairs, rank-major) is the
// plan's choice; the kernel walks the plan's task list. The tiles of that
// list go to the persistent units (CTAs or CTA pairs) round-robin; under the
// tail split the last waves are dealt out as equal k-block ranges instead
// (get_work).
//
// Two tile configurations:
//   PAIR = false  one CTA per SM owns a 128 x 256 fp32 accumulator; the MMA
//                 is tcgen05.mma.cta_group::1 (M = 128, N = 256).
//   PAIR = true   a cluster of two CTAs (two SMs) owns a 256 x 256 tile:
//                 each CTA loads 128 rows of A and 128 columns of B, the
//                 leader issues tcgen05.mma.cta_group::2 (M = 256, N = 256)
//                 reading both CTAs' shared memory, and each CTA's TMEM holds
//                 its 128 rows x 256 columns. Operand traffic into each SM
//                 is 2/3 of the single-CTA tile's.
//
// Warp roles (192 threads per CTA; 320 with movers):
//   warp 0     TMA producer: 128-byte-wide K slices of both operands into a
//              shared-memory ring (128B swizzle); 4 stages of 48 KB, or 6 of
//              32 KB per CTA in the pair.
//   warp 1     allocates 512 TMEM columns (two fp32 accumulators); in the
//              single-CTA kernel and in the pair's leader it issues the MMAs.
//   warps 2-5  epilogue: tcgen05.ld the accumulator (each warp its 32-lane
//              quarter), stage 32-row sub-tiles in shared memory, move them
//              with TMA:
//                RS/DP  the partial of chunk c goes to owner c's shard: the
//                       first partial of a shard tile is stored, later ones
//                       are added (TMA reduce-add, fp32, at L2) once the
//                       per-tile counter says the shard holds the first. This
//                       accumulate is the P2P transfer. With a completion
//                       action (bf16 output, all-reduce) the owner's last
//                       partial finishes the tile; under the ring RS each
//                       later hop adds the running sum its predecessor
//                       forwarded and passes the result on.
//                AG     bf16 store into rank r's output rows of the source
//                       shard; the A operand was read straight from the
//                       source rank's buffer (the transfer is the read), or
//                       from r's gather buffer under the copy transport.
//                       All-to-all (same kernel): X_r times W_r's column
//                       block c, stored into rank c's output at rank r's
//                       rows (the transfer is the store).
//                PARTIAL fp32 store into the computing rank's own buffer
//                       (pure-GEMM control, no transfer).
//   warps 6-9  (MOV) movers: 128-bit copies of 32-row shard pieces into the
//              gather buffers, ring-forwarded behind ready flags (copy
//              transport) or as a side output (peer read, wide outputs).
//              With narrow outputs under peer read, the producer instead
//              stores the A stages it loaded into the gather buffers.
// Synchronisation (shd-paper.top, 方法详解 "key design" paragraph, item 3):
// mbarriers inside the CTA / pair, acquire/release counters and flags in
// global memory across CTAs; every wait is bounded and failures land in a
// status word. Optional %globaltimer stamps per CTA record when its math and
// its transfers ended.
#pragma once

#include "fo_device.cuh"
#include "fo_internal.h"

namespace fo {

constexpr int kEpiWarps = 4;
constexpr int kEpiBuf = 32 * 128;              // 32 rows x 128 bytes
// Staging buffers per epilogue warp and pipeline depths (overridable at
// build time; the defaults fill the 227 KB of shared memory). The short-
// reduction variant (SK) of the CTA-pair kernel trades a pipeline stage for
// two more staging buffers per warp: with few k-blocks per tile the
// epilogue, not the operand stream, sets the pace.
#ifndef FO_EPI_BUFS
#define FO_EPI_BUFS 2
#endif
#ifndef FO_PAIR_STAGES
#define FO_PAIR_STAGES 6
#endif
#ifndef FO_SINGLE_STAGES
#define FO_SINGLE_STAGES 4
#endif
#ifndef FO_SK_EPI_BUFS
#define FO_SK_EPI_BUFS 4
#endif
#ifndef FO_SK_PAIR_STAGES
#define FO_SK_PAIR_STAGES 5
#endif
constexpr int kThreads = 32 * (2 + kEpiWarps);
// AG variants that also move X shards into the gather buffers G_r carry four
// more warps; a piece is 32 rows of one shard.
constexpr int kMoverWarps = 4;
constexpr int kPieceRows = 32;
__host__ __device__ constexpr int threads_for(bool movers) { return 32 * (2 + kEpiWarps + (movers ? kMoverWarps : 0)); }
constexpr int kBarBytes = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kMbarLimitNs = 2000000000ull;

template <bool PAIR, bool SK = false>
struct Cfg {
  static_assert(!SK || PAIR, "the short-reduction variant has CTA-pair tiles");
  static constexpr int kStages = PAIR ? (SK ? FO_SK_PAIR_STAGES : FO_PAIR_STAGES) : FO_SINGLE_STAGES;
  static constexpr int kEpiBufs = SK ? FO_SK_EPI_BUFS : FO_EPI_BUFS;
  static constexpr int kAStage = FO_BM * FO_BK_BYTES;                       // 16 KB
  static constexpr int kBRows = PAIR ? FO_BN / 2 : FO_BN;                   // B rows (N) in this CTA
  static constexpr int kBStage = kBRows * FO_BK_BYTES;                      // 16 or 32 KB
  static constexpr int kStageBytes = kAStage + kBStage;
  static constexpr int kTileM = PAIR ? 2 * FO_BM : FO_BM;                   // rows of one tile
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kEpiWarps * kEpiBufs * kEpiBuf + kBarBytes;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

enum Epi : int { EPI_RS = 0, EPI_AG = 1, EPI_PARTIAL = 2 };

struct alignas(128) FoParams {
  CUtensorMap tmA[FO_MAX_R];   // RS: X_r; DP: X_r ([T x M]); AG: X_src
  CUtensorMap tmB[FO_MAX_R];   // W_r or dY_r
  CUtensorMap tmD[FO_MAX_R];   // RS/DP: Y_c (2-D); AG: Y_r (3-D); PARTIAL: P_r (3-D)
  int32_t table[FO_MAX_R][FO_MAX_R];
  int32_t ord[FO_MAX_R][FO_MAX_R];
  int32_t task_r[FO_MAX_R * FO_MAX_R];   // rank and step of the i-th chunk task in execution order
  int32_t task_s[FO_MAX_R * FO_MAX_R];
  int32_t R;
  int32_t tiles_m;             // m-tiles per chunk, of this kernel's tile height (128 or 256 rows)
  int32_t tiles_n;
  int32_t num_kb;
  int32_t rows_per_chunk;
  int32_t deterministic;
  int32_t fault_inject;
  int32_t ctr_tiles_m;         // 128-row tiles per chunk in the counter array
  uint32_t* counters;          // RS/DP: [R][ctr_tiles_m][tiles_n][4]
  int32_t* status;             // fo_ws_header
  uint64_t timeout_ns;
  // AG with a gather buffer (movers):
  CUtensorMap tmG[FO_MAX_R];   // G_r [M x K]: the A operand of steps >= 1 under the copy transport
  const void* xsrc[FO_MAX_R];  // X_r
  void* gdst[FO_MAX_R];        // G_r
  uint32_t* flags;             // copy transport: ready flags [R][R][pieces]
  uint32_t* epoch;             // fo_ws_header::epoch (exit_count follows)
  int64_t row_bytes;           // K * 2
  int32_t pieces;              // 32-row pieces per shard
  int32_t ag_copy;             // 1: shards reach G_r along the ring and the GEMM reads them there
  // All-to-all (EPI_AG kernels): task (r, s) multiplies X_r by column block
  // c = table[r][s] of W_r (columns c * n_cols ...) and stores the bf16 tile
  // into rank c's output at rank r's rows (tmD[c] viewed [n_cols, rows/R, R]).
  int32_t a2a;
  // (GST kernels: tmG views G_r as [K, rows/R, R], the map of the stores.)
  // RS/DP completion: the owner's last partial (contribution R-1) is the
  // finisher. It waits for the other R-1, adds their sum (read from the
  // shard rows tmD[c] addresses) to its own partial and writes the result:
  int32_t completion;          // FO_COMPLETE_*
  int64_t n_cols;              // N: columns of a shard row
  float* shard[FO_MAX_R];      // fp32 shard rows that tmD[c] addresses
  CUtensorMap tmF[FO_MAX_R];   // BF16: the bf16 shard outputs [rows/R x N] (2-D)
  CUtensorMap tmAR[FO_MAX_R];  // ALLREDUCE: every rank's full output as [N, rows/R, R] (3-D);
                               // ring RS: every rank's receive buffer, same shape
  // Ring RS: the partial of hop s > 0 (the s-th rank of chunk c's chain) is
  // added to the running sum its predecessor left in inbox[r] (chunk c's
  // rows) and forwarded into inbox[r+1], or, at the last hop (the owner),
  // written to the output.
  int32_t ring;
  float* inbox[FO_MAX_R];      // rank q's receive buffer [M x N] fp32 (chunk-major rows)
  // Tracing: FO_TRACE_STAMPS %globaltimer stamps per CTA (null: off).
  uint64_t* trace;
  // Fault injection: tiles of the first task wait this long after their
  // CTA started before their operands are loaded (0: off).
  uint64_t delay_ns;
  // Tail split: the last sk_tiles tiles of the launch (the last partial
  // wave plus up to two whole waves) are cut along K so that every unit gets the
  // same number of k-blocks (0: off). A cut tile's head part leaves its fp32
  // partial in the split buffer (tmSK / sk_buf, one kTileM x FO_BN block
  // per split tile) and releases sk_ctr[(tile * 2 + cta) * 4 + quarter];
  // its finishing part adds it and completes the tile as usual.
  int32_t sk_tiles;
  float* sk_buf;
  uint32_t* sk_ctr;
  CUtensorMap tmSK;
  // MN-major A given as R row shards of a_shard_rows rows each (0: one A per
  // rank): the rows of k-block kb come from shard kb * kBK / a_shard_rows,
  // whose map is tmA[shard]. Every task reads the same A, in place: the
  // all-gather of the shards, without a gathered copy.
  int32_t a_shard_rows;
};

enum Completion : int { FO_COMPLETE_NONE = 0, FO_COMPLETE_BF16 = 1, FO_COMPLETE_ALLREDUCE = 2 };

template <bool A_MN, bool B_MN, bool TF32, bool PAIR>
__host__ __device__ constexpr uint32_t instr_desc() {
  // kind::f16 / kind::tf32 instruction descriptor: D fp32 (bits 4-5 = 1),
  // A and B format (bits 7-9, 10-12: bf16 = 1, tf32 = 2), A/B major (bits 15,
  // 16: 1 = MN-major), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
  return (1u << 4) | ((TF32 ? 2u : 1u) << 7) | ((TF32 ? 2u : 1u) << 10) | ((A_MN ? 1u : 0u) << 15) |
         ((B_MN ? 1u : 0u) << 16) | ((uint32_t)(FO_BN >> 3) << 17) |
         ((uint32_t)((PAIR ? 2 * FO_BM : FO_BM) >> 4) << 24);
}

struct Tile {
  int r, s, c, ord, mt, nt;    // mt: m-tile of this kernel's tile height
};

// One unit of a CTA's (or CTA pair's) work: k-blocks [kb0, kb1) of tile L.
// FULL covers the whole reduction. Under the tail split a tile may be cut
// once: its HEAD part (from k-block 0) leaves an fp32 partial, its FINISH
// part (to the last k-block) adds that partial and completes the tile.
enum WorkRole : int { WORK_FULL = 0, WORK_HEAD = 1, WORK_FINISH = 2 };
struct Work {
  int L, kb0, kb1, role, sk;   // sk: index among the split tiles (HEAD / FINISH)
};

// The i-th work item of `unit` (false when there is none). Without the tail
// split, tiles go round-robin: unit, unit + units, ... With it, the first
// total - sk_tiles tiles (whole waves) go round-robin, and the k-blocks of
// the last sk_tiles tiles are dealt out in equal contiguous ranges, each at
// least one tile long, so a tile is cut at most once. Every unit runs its
// HEAD part first: a HEAD never waits, so each FINISH waits only for work
// that runs ahead of anything it could block.
__device__ __forceinline__ bool get_work(const FoParams& p, int total, int unit, int units, int i, Work& w) {
  const int nkb = p.num_kb;
  if (p.sk_tiles == 0) {
    const int L = unit + i * units;
    if (L >= total) return false;
    w.L = L, w.kb0 = 0, w.kb1 = nkb, w.role = WORK_FULL, w.sk = -1;
    return true;
  }
  const int first = total - p.sk_tiles;   // a whole number of waves
  const int ndp = first / units;
  if (i < ndp) {
    w.L = unit + i * units, w.kb0 = 0, w.kb1 = nkb, w.role = WORK_FULL, w.sk = -1;
    return true;
  }
  const int j = i - ndp;
  const int64_t iters = (int64_t)p.sk_tiles * nkb;
  const int64_t a = iters * unit / units, b = iters * (unit + 1) / units;
  if (a >= b) return false;
  const int ta = (int)(a / nkb), tb = (int)((b - 1) / nkb);
  const int nseg = tb - ta + 1;
  if (j >= nseg) return false;
  const int kb1_last = (int)((b - 1) % nkb) + 1;
  const bool head_last = nseg > 1 && kb1_last < nkb;   // the range ends inside tile tb
  const int kseg = head_last ? (j == 0 ? nseg - 1 : j - 1) : j;
  w.sk = ta + kseg;
  w.L = first + w.sk;
  w.kb0 = kseg == 0 ? (int)(a % nkb) : 0;
  w.kb1 = kseg == nseg - 1 ? kb1_last : nkb;
  w.role = (w.kb0 == 0 && w.kb1 == nkb) ? WORK_FULL : (w.kb0 == 0 ? WORK_HEAD : WORK_FINISH);
  return true;
}

__device__ __forceinline__ Tile decode_tile(const FoParams& p, int L) {
  const int tpt = p.tiles_m * p.tiles_n;
  const int task = L / tpt;
  const int t = L - task * tpt;
  Tile ti;
  ti.s = p.task_s[task];
  ti.r = p.task_r[task];
  ti.mt = t / p.tiles_n;
  ti.nt = t - ti.mt * p.tiles_n;
  ti.c = p.table[ti.r][ti.s];
  ti.ord = p.ord[ti.r][ti.s];
  return ti;
}

// A partial is in its owner's shard: count it. The partial that completes
// the shard (the R-th) resets the counter for the next call.
// Returns true for the partial that completes the tile (it also acquires
// every other partial's release, so the completed tile can be read).
__device__ __forceinline__ bool signal_partial(uint32_t* ctr, int R) {
  const uint32_t old = atom_add_acq_rel_u32(ctr, 1u);
  if (old + 1u == (uint32_t)R) {
    atomicExch(ctr, 0u);
    return true;
  }
  return false;
}

// Copy n16 16-byte words with nthr threads (thread tid handles words tid,
// tid + nthr, ...), sixteen loads in flight per thread (the four mover warps
// of a CTA keep 32 KB in flight; eight loads left the gather copies
// latency-bound); L2-only caching.
__device__ __forceinline__ void copy16(const uint8_t* from, uint8_t* to, size_t n16, int tid, int nthr) {
  const uint4* s = reinterpret_cast<const uint4*>(from);
  uint4* d = reinterpret_cast<uint4*>(to);
  constexpr int U = 16;
  size_t i = (size_t)tid;
  for (; i + (size_t)(U - 1) * nthr < n16; i += (size_t)U * nthr) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = __ldcg(s + i + (size_t)u * nthr);
#pragma unroll
    for (int u = 0; u < U; ++u) __stcg(d + i + (size_t)u * nthr, v[u]);
  }
  for (; i < n16; i += nthr) __stcg(d + i, __ldcg(s + i));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Write 32 registers (one 128-byte row per thread) into a 32 x 128 B staging
// buffer in the TMA 128B-swizzle layout: 16-byte chunk j of row i lives at
// chunk j ^ (i % 8).
__device__ __forceinline__ void stage_row_sw128(uint32_t buf, int lane, const uint32_t (&w)[32]) {
  const uint32_t row = buf + (uint32_t)lane * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t addr = row + ((uint32_t)(j ^ (lane & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[4 * j]), "r"(w[4 * j + 1]),
                 "r"(w[4 * j + 2]), "r"(w[4 * j + 3])
                 : "memory");
  }
}

// Coalesced loads of the 32 x 32 fp32 block at (row0, col0) of a [rows x
// ncols] row-major matrix with leading dimension ld: lane l loads the
// 16-byte chunk l % 8 of rows row0 + l / 8 + 4 i (i = 0..7), four whole
// 128-byte rows per instruction. Rows past `rows`, columns past `ncols` or
// a null matrix read as zero.
__device__ __forceinline__ void load_block32_coalesced(const float* src, int row0, int rows, int col0, int ncols,
                                                       size_t ld, int lane, float4 (&sv)[8]) {
  const int crow = lane >> 3, col = col0 + (lane & 7) * 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = row0 + 4 * i + crow;
    sv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (src && row < rows && col < ncols) sv[i] = __ldcg(reinterpret_cast<const float4*>(src + (size_t)row * ld + col));
  }
}

// Adds a block loaded by load_block32_coalesced into a 32 x 128 B fp32
// staging buffer in the 128B-swizzle layout (stage_row_sw128).
__device__ __forceinline__ void add_block32_sw128(uint32_t buf, int lane, const float4 (&sv)[8]) {
  const int crow = lane >> 3, cch = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = 4 * i + crow;
    const uint32_t a = buf + (uint32_t)rr * 128u + ((uint32_t)(cch ^ (rr & 7)) << 4);
    float4 x;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                 : "r"(a)
                 : "memory");
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x.x + sv[i].x), "f"(x.y + sv[i].y),
                 "f"(x.z + sv[i].z), "f"(x.w + sv[i].w)
                 : "memory");
  }
}

// Reads row `lane` (32 fp32) back from a staging buffer in the 128B-swizzle
// layout.
__device__ __forceinline__ void read_row_sw128(uint32_t buf, int lane, float (&f)[32]) {
  const uint32_t row = buf + (uint32_t)lane * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = row + ((uint32_t)(j ^ (lane & 7)) << 4);
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(f[4 * j]), "=f"(f[4 * j + 1]), "=f"(f[4 * j + 2]), "=f"(f[4 * j + 3])
                 : "r"(a)
                 : "memory");
  }
}

// GST: peer-read all-gather with a gather buffer and narrow outputs: the
// producer writes every A stage it loaded for a tile of the first column
// block back out to G_r, instead of mover warps copying the shards.
template <int EPI, bool A_MN, bool B_MN, bool TF32, bool PAIR, bool MOV = false, bool GST = false, bool SK = false>
__global__ void __launch_bounds__(threads_for(MOV), 1) fo_chunk_gemm_kernel(const __grid_constant__ FoParams p) {
  static_assert(!MOV || EPI == EPI_AG, "movers belong to the all-gather kernel");
  static_assert(!GST || (EPI == EPI_AG && !MOV), "gather stores replace the movers of the all-gather kernel");
  using C = Cfg<PAIR, SK>;
  constexpr int kEpiBufs = C::kEpiBufs;
  constexpr int CG = PAIR ? 2 : 1;
  constexpr int kStages = C::kStages;
  constexpr int kEsz = TF32 ? 4 : 2;
  constexpr int kBK = FO_BK_BYTES / kEsz;        // K elements per stage (= MN elements per 128B row)
  constexpr int kMmaK = 32 / kEsz;               // K of one tcgen05.mma (32 bytes)
  constexpr int kBoxBytes = kBK * 128;           // one MN-major box: kBK rows x 128 B
  constexpr uint32_t kIdesc = instr_desc<A_MN, B_MN, TF32, PAIR>();
  constexpr uint32_t kTxBytes = (PAIR ? 2 : 1) * C::kStageBytes;   // both halves land on the leader's barrier

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sStage = base;
  const uint32_t sEpi = base + kStages * C::kStageBytes;
  const uint32_t sBar = sEpi + kEpiWarps * kEpiBufs * kEpiBuf;
  auto full_bar = [&](int i) { return sBar + 8u * i; };
  auto empty_bar = [&](int i) { return sBar + 8u * (kStages + i); };
  auto tfull_bar = [&](int a) { return sBar + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return sBar + 8u * (2 * kStages + 2 + a); };
  const uint32_t mma_done_bar = sBar + 8u * (2 * kStages + 4);
  const uint32_t sTmemSlot = sBar + 8u * (2 * kStages + 5);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + (sTmemSlot - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (sTmemSlot - base) + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const volatile int32_t* gstatus = p.status;
  // Position in the pair (0 = leader) and the pair's index; a single-CTA
  // kernel is its own leader.
  const uint32_t prank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const bool leader = prank == 0;
  // Launch epoch of the copy transport's ready flags (read before this CTA
  // can count itself out; the last CTA of the launch advances it).
  const uint32_t epoch0 = MOV ? *reinterpret_cast<volatile uint32_t*>(p.epoch) : 0u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  const uint64_t t_start = globaltimer();
  uint64_t* const trace = (p.trace && blockIdx.x < FO_TRACE_MAX_CTAS) ? p.trace + (size_t)blockIdx.x * FO_TRACE_STAMPS
                                                                       : nullptr;
  if (trace && threadIdx.x == 0) {
    trace[0] = t_start;
    for (int i = 1; i < FO_TRACE_STAMPS; ++i) trace[i] = 0;
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc<CG>(sTmemSlot, kTmemCols);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();   // the peer's barriers are initialised before any remote arrive
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = p.R * p.R * p.tiles_m * p.tiles_n;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t it = 0;
      // The ring position of k-block `it`, stepped along with it: the
      // producer's path from a freed stage to its next loads is the MMA's
      // critical path, so it carries no division.
      int pst = 0;
      uint32_t pph = 0;
      // All-gather: the X shards, which every rank's tasks read again, stay
      // in L2 ahead of the streamed outputs.
      const uint64_t pol_x = l2_policy_evict_last();
      // Gather stores still owed per stage: the A block a stage holds goes to
      // G_r once the MMA has read it and before the stage is refilled.
      constexpr int kG = GST ? kStages : 1;
      int g_r[kG], g_c[kG] = {}, g_row[kG] = {}, g_k[kG] = {};
      uint32_t g_it[kG] = {};
#pragma unroll
      for (int i = 0; i < kG; ++i) g_r[i] = -1;
      auto g_flush = [&](int st) {
        if constexpr (GST) {
          if (g_r[st] >= 0) {
            tma_store_3d(&p.tmG[g_r[st]], sStage + st * C::kStageBytes, g_k[st], g_row[st], g_c[st]);
            bulk_commit();
            bulk_wait_read<0>();   // the stage may be refilled once the store has read it
            g_r[st] = -1;
          }
        }
      };
      Work w;
      // Another CTA's recorded failure ends this one's work. The status word
      // is read at a tile's start and tested at the next one's, so its
      // global round trip never holds up the tile's first loads.
      int32_t gs = 0;
      for (int wi = 0; get_work(p, total, unit, units, wi, w); ++wi) {
        const int L = w.L;
        if (gs) *abort_flag = 1;
        if (*abort_flag) break;
        gs = *gstatus;
        const Tile ti = decode_tile(p, L);
        if (p.delay_ns && L < p.tiles_m * p.tiles_n) {
          // Fault injection: hold the first task's tiles (bounded by the
          // delay itself; an abort ends it early).
          while (globaltimer() - t_start < p.delay_ns && !*abort_flag && !*gstatus) __nanosleep(2000);
        }
        const CUtensorMap* mA = EPI == EPI_AG ? &p.tmA[p.a2a ? ti.r : ti.c] : &p.tmA[ti.r];
        const CUtensorMap* mB = &p.tmB[ti.r];
        // Row (or column, for MN-major A) where this CTA's A block starts,
        // and the first output column of its B block (in the all-to-all,
        // within W_r's column block c).
        int a_mn0 = (EPI == EPI_AG ? 0 : ti.c * p.rows_per_chunk) + ti.mt * C::kTileM + (int)prank * FO_BM;
        const int b_n0 = (EPI == EPI_AG && p.a2a ? ti.c * (int)p.n_cols : 0) + ti.nt * FO_BN + (int)prank * C::kBRows;
        if constexpr (MOV) {
          if (p.ag_copy && ti.s > 0) {
            // Copy transport: this shard reached G_r along the ring. Wait
            // until the pieces holding this CTA's 128 rows are ready.
            const int r0 = ti.mt * C::kTileM + (int)prank * FO_BM;
            const int p0 = r0 / kPieceRows;
            const int p1 = min(p.pieces, (r0 + FO_BM + kPieceRows - 1) / kPieceRows);
            bool good = true;
            for (int pc = p0; pc < p1 && good; ++pc)
              good = wait_flag_eq(&p.flags[((size_t)ti.r * p.R + ti.c) * p.pieces + pc], epoch0 + 1u, p.timeout_ns,
                                  abort_flag, gstatus);
            if (!good) {
              if (!*abort_flag && !*gstatus) record_error(p.status, FO_ERR_TIMEOUT, ti.r, ti.s, ti.c);
              *abort_flag = 1;
              break;
            }
            fence_proxy_async_global();
            mA = &p.tmG[ti.r];
            a_mn0 = ti.c * p.rows_per_chunk + r0;
          }
        }
        bool ok = true;
        // Sharded A: the shard of the task's first k-block, then stepped
        // along with the k-blocks (no division in the loop).
        int a_src = 0, a_base = 0;
        if constexpr (A_MN) {
          if (p.a_shard_rows) {
            a_src = (w.kb0 * kBK) / p.a_shard_rows;
            a_base = a_src * p.a_shard_rows;
          }
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int stage = pst;
          const uint32_t ph = pph;
          if (++pst == kStages) {
            pst = 0;
            pph ^= 1u;
          }
          if (!mbar_wait(empty_bar(stage), ph ^ 1u, abort_flag, kMbarLimitNs)) {
            ok = false;
            break;
          }
          g_flush(stage);
          const uint32_t sa = sStage + stage * C::kStageBytes;
          const uint32_t sb = sa + C::kAStage;
          const int k0 = kb * kBK;
          if constexpr (GST) {
            if (ti.nt == 0) {
              g_r[stage] = ti.r, g_c[stage] = ti.c, g_row[stage] = a_mn0, g_k[stage] = k0, g_it[stage] = it;
            }
          }
          // A given as row shards: this k-block's rows are in one shard.
          const CUtensorMap* mAk = mA;
          int kA = k0;
          if constexpr (A_MN) {
            if (p.a_shard_rows) {
              if (k0 - a_base >= p.a_shard_rows) {
                ++a_src;
                a_base += p.a_shard_rows;
              }
              kA = k0 - a_base;
              mAk = &p.tmA[a_src];
            }
          }
          if constexpr (PAIR) {
            const uint32_t fb = mapa_shared(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), kTxBytes);
            if constexpr (A_MN) {
#pragma unroll
              for (int j = 0; j < FO_BM / kBK; ++j) tma_load_2d_pair(sa + j * kBoxBytes, mAk, fb, a_mn0 + j * kBK, kA);
            } else {
              if (EPI == EPI_AG) tma_load_2d_pair_hint(sa, mA, fb, k0, a_mn0, pol_x);
              else tma_load_2d_pair(sa, mA, fb, k0, a_mn0);
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int j = 0; j < C::kBRows / kBK; ++j)
                tma_load_2d_pair(sb + j * kBoxBytes, mB, fb, b_n0 + j * kBK, k0);
            } else {
              tma_load_2d_pair(sb, mB, fb, k0, b_n0);
            }
          } else {
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, kTxBytes);
            if constexpr (A_MN) {
#pragma unroll
              for (int j = 0; j < FO_BM / kBK; ++j) tma_load_2d(sa + j * kBoxBytes, mAk, fb, a_mn0 + j * kBK, kA);
            } else {
              if (EPI == EPI_AG) tma_load_2d_hint(sa, mA, fb, k0, a_mn0, pol_x);
              else tma_load_2d(sa, mA, fb, k0, a_mn0);
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int j = 0; j < C::kBRows / kBK; ++j) tma_load_2d(sb + j * kBoxBytes, mB, fb, b_n0 + j * kBK, k0);
            } else {
              tma_load_2d(sb, mB, fb, k0, b_n0);
            }
          }
        }
        if (!ok) break;
      }
      // Gather stores still owed: each waits until the MMA has read its stage.
      if constexpr (GST) {
        if (!*abort_flag) {
#pragma unroll 1
          for (int st = 0; st < kStages; ++st) {
            if (g_r[st] < 0) continue;
            if (!mbar_wait(empty_bar(st), (g_it[st] / kStages) & 1u, abort_flag, kMbarLimitNs)) break;
            g_flush(st);
          }
        }
        bulk_wait<0>();
      }
      // Drain: every load still in flight lands before the CTA may exit.
      // The pair's loads complete on the leader's barriers, which count both
      // halves; after an abort the peer gives its own loads a fixed time.
      volatile int never = 0;
      if (leader) {
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait(full_bar(j % kStages), (j / kStages) & 1u, &never, 100000000ull);
      } else if (*abort_flag) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
      }
      if (*abort_flag) record_error(p.status, FO_ERR_TIMEOUT, -1, -1, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      uint32_t it = 0, tcount = 0;
      int mst = 0;   // ring position of k-block `it`, stepped along with it
      uint32_t mph = 0;
      Work w;
      for (int wi = 0; get_work(p, total, unit, units, wi, w); ++wi, ++tcount) {
        if (*abort_flag) break;
        const int acc = tcount & 1;
        const uint32_t aph = (tcount >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, kMbarLimitNs)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * FO_BN);
        bool ok = true;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int stage = mst;
          const uint32_t ph = mph;
          if (++mst == kStages) {
            mst = 0;
            mph ^= 1u;
          }
          if (!mbar_wait(full_bar(stage), ph, abort_flag, kMbarLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sStage + stage * C::kStageBytes;
          const uint32_t sb = sa + C::kAStage;
#pragma unroll
          for (int k = 0; k < FO_BK_BYTES / 32; ++k) {
            // K-major: the k-th 32-byte column of the swizzled 128-byte rows.
            // MN-major: kMmaK K-rows of 128 bytes further into each box.
            const uint32_t aoff = A_MN ? (uint32_t)(k * kMmaK * 128) : (uint32_t)(k * 32);
            const uint32_t boff = B_MN ? (uint32_t)(k * kMmaK * 128) : (uint32_t)(k * 32);
            const uint64_t adesc =
                A_MN ? smem_desc_sw128(sa + aoff, kBoxBytes, 1024) : smem_desc_sw128(sa + aoff, 16, 1024);
            const uint64_t bdesc =
                B_MN ? smem_desc_sw128(sb + boff, kBoxBytes, 1024) : smem_desc_sw128(sb + boff, 16, 1024);
            tc_mma<CG, TF32>(d, adesc, bdesc, kIdesc, (kb != w.kb0 || k != 0) ? 1u : 0u);
          }
          if constexpr (PAIR) tc_commit_pair_multicast(empty_bar(stage), 0x3);
          else tc_commit<1>(empty_bar(stage));
        }
        if (!ok) break;
        if constexpr (PAIR) tc_commit_pair_multicast(tfull_bar(acc), 0x3);
        else tc_commit<1>(tfull_bar(acc));
      }
      // All issued MMAs complete before TMEM is released.
      tc_commit<CG>(mma_done_bar);
      volatile int never = 0;
      mbar_wait(mma_done_bar, 0, &never, 100000000ull);
      if (trace) trace[1] = globaltimer();
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;        // staging buffers of this warp
    const int q = warp & 3;        // TMEM lane quarter this warp may access
    uint32_t tcount = 0;
    constexpr int kSubRS = FO_BN / 32;   // bulk groups per RS tile quarter
    // RS: this warp's last partial, not yet published (same in every lane).
    uint32_t* pend_ctr = nullptr;
    bool pend_skip = false;
    // Publish the deferred partial (every lane calls; lane 0 owns the bulk
    // groups): wait until its writes are performed (all groups, or all but
    // the newest tile's 8) and release-count it.
    auto publish = [&](bool all) {
      if (!pend_ctr) return;
      if (lane == 0) {
        if (all) bulk_wait<0>();
        else bulk_wait<kSubRS>();
        fence_proxy_async_global();
        if (!pend_skip) signal_partial(pend_ctr, p.R);
      }
      pend_ctr = nullptr;
    };
    Work w;
    for (int wi = 0; get_work(p, total, unit, units, wi, w); ++wi, ++tcount) {
      if (*abort_flag) break;
      const Tile ti = decode_tile(p, w.L);
      const int acc = tcount & 1;
      const uint32_t aph = (tcount >> 1) & 1u;
      // Tiles of the split region run close together on every unit, so a
      // partial another tile may wait for is released at once, not a tile
      // later.
      const bool in_split = p.sk_tiles != 0 && w.L >= total - p.sk_tiles;
      if constexpr (EPI == EPI_RS) {
        if (p.ring && ti.ord > 0 && w.role != WORK_HEAD) {
          // Ring hop: warm L2 with the running sum this warp will read once
          // the accumulator is ready (each lane one row of its quarter).
          const int row = (ti.mt * (PAIR ? 2 : 1) + (int)prank) * FO_BM + q * 32 + lane;
          const int ncol = min(FO_BN, (int)p.n_cols - ti.nt * FO_BN);
          if (row < p.rows_per_chunk && ncol > 0)
            prefetch_l2_bulk(p.inbox[ti.r] + ((size_t)ti.c * p.rows_per_chunk + row) * (size_t)p.n_cols +
                                 (size_t)ti.nt * FO_BN,
                             (uint32_t)ncol * 4u);
        }
        // About to block until the next accumulator is ready: publish the
        // deferred partial first (a warp never holds one while it waits, so
        // a waiter elsewhere always sees it eventually).
        const uint32_t ready = (lane == 0 && pend_ctr) ? mbar_try_wait(tfull_bar(acc), aph) : 1u;
        if (!__shfl_sync(0xffffffffu, ready, 0)) publish(true);
      }
      if (!mbar_wait(tfull_bar(acc), aph, abort_flag, kMbarLimitNs)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * FO_BN);
      const int mt128 = ti.mt * (PAIR ? 2 : 1) + (int)prank;   // 128-row tile of this CTA within the chunk
      const int row0 = mt128 * FO_BM + q * 32;                   // first row of this quarter within the chunk
      const int n0 = ti.nt * FO_BN;

      if (w.role != WORK_FULL) {
        // Tail split. This warp's 32 rows of the tile in the split buffer:
        const int srow = w.sk * C::kTileM + (int)prank * FO_BM + q * 32;
        uint32_t* const sc = p.sk_ctr + ((size_t)w.sk * 2 + prank) * 4 + q;
        constexpr int kSub = FO_BN / 32;
        if (w.role == WORK_HEAD) {
          // Head part: store the fp32 partial, free the accumulator and
          // release the partial to the finishing part.
          // (At most one head and one finishing part per unit and launch.
          // The loops handle two sub-tiles per trip with fixed registers:
          // the second's loads are in flight while the first is processed.)
          if constexpr (EPI == EPI_RS) publish(true);
          auto head_store = [&](int j, uint32_t(&v)[32]) {
            const uint32_t buf = sEpi + (uint32_t)((e * kEpiBufs + (j % kEpiBufs)) * kEpiBuf);
            if (lane == 0) bulk_wait_read<kEpiBufs - 1>();
            __syncwarp();
            stage_row_sw128(buf, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.tmSK, buf, j * 32, srow);
              bulk_commit();
            }
          };
#pragma unroll 1
          for (int j = 0; j < kSub; j += 2) {
            uint32_t va[32], vb[32];
            tmem_ld32(tbase + j * 32, va);
            tmem_ld32(tbase + (j + 1) * 32, vb);
            tmem_ld_wait();
            reg_fence(va);
            reg_fence(vb);
            if (j + 2 == kSub) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
                else mbar_arrive(tempty_bar(acc));
              }
            }
            head_store(j, va);
            head_store(j + 1, vb);
          }
          if (lane == 0) {
            bulk_wait<0>();
            fence_proxy_async_global();
            atom_add_release_u32(sc, 1u);
          }
          __syncwarp();
          continue;
        }
        // Finishing part: wait for the head part's partial and add it into
        // the accumulator; the tile then completes like any other.
        int good = 1;
        const uint32_t have = __shfl_sync(0xffffffffu, lane == 0 ? ld_acquire_u32(sc) : 0u, 0);
        if (have < 1u) {
          if constexpr (EPI == EPI_RS) publish(true);
          if (lane == 0) {
            good = wait_counter_geq(sc, 1u, p.timeout_ns, abort_flag, gstatus) ? 1 : 0;
            if (!good && !*abort_flag && !*gstatus) record_error(p.status, FO_ERR_TIMEOUT, ti.r, ti.s, ti.c);
          }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t abuf = sEpi + (uint32_t)(e * kEpiBufs * kEpiBuf);
        const int srows = (w.sk + 1) * C::kTileM;
        if (lane == 0) bulk_wait_read<0>();   // no store still reads the staging buffer
        __syncwarp();
        auto finish_add = [&](int j, const float4(&hs)[8]) {
          uint32_t v[32];
          tmem_ld32(tbase + j * 32, v);
          tmem_ld_wait();
          reg_fence(v);
          stage_row_sw128(abuf, lane, v);
          __syncwarp();
          add_block32_sw128(abuf, lane, hs);
          __syncwarp();
          float f[32];
          read_row_sw128(abuf, lane, f);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(f[i]);
          tmem_st32(tbase + j * 32, v);
          __syncwarp();   // every lane has read its row before the next sub-tile is staged
        };
        float4 ha[8], hb[8];
        load_block32_coalesced(p.sk_buf, srow, srows, 0, FO_BN, FO_BN, lane, ha);
        load_block32_coalesced(p.sk_buf, srow, srows, 32, FO_BN, FO_BN, lane, hb);
#pragma unroll 1
        for (int j = 0; j < kSub; j += 2) {
          finish_add(j, ha);
          if (j + 2 < kSub) load_block32_coalesced(p.sk_buf, srow, srows, (j + 2) * 32, FO_BN, FO_BN, lane, ha);
          finish_add(j + 1, hb);
          if (j + 3 < kSub) load_block32_coalesced(p.sk_buf, srow, srows, (j + 3) * 32, FO_BN, FO_BN, lane, hb);
        }
        tmem_st_wait();
        if (lane == 0) atomicExch(sc, 0u);   // consumed: ready for the next launch
        __syncwarp();
      }

      uint32_t* ctr = nullptr;
      bool ok = true;
      // The owner's last partial finishes the tile when the plan has a
      // completion action (all-reduce, bf16 output). Under the ring RS every
      // later hop of a chain is a finisher too: it adds the running sum its
      // predecessor forwarded and passes the result on.
      const bool last = ti.ord == p.R - 1;
      const bool ring = EPI == EPI_RS && p.ring != 0;
      const bool hop = ring && ti.ord > 0;
      const bool fin = EPI == EPI_RS && ((p.completion != FO_COMPLETE_NONE && last) || hop);
      if constexpr (EPI == EPI_RS) {
        ctr = p.counters + (((size_t)ti.c * p.ctr_tiles_m + mt128) * p.tiles_n + ti.nt) * 4 + q;
        // A bf16 finisher commits 4 bulk groups per tile, not a reduce
        // tile's 8: release the pending partial before it. A ring hop
        // releases its predecessor tile's forward here too: the next hop
        // of that chain may be only a tile behind.
        if (fin && (hop || (last && p.completion == FO_COMPLETE_BF16))) publish(true);
        if (ti.ord > 0) {
          // The shard must already hold its first (stored) partial; in
          // deterministic mode every partial before this one; the finisher
          // needs all R-1 others; a ring hop needs its predecessor's forward
          // (hop ord-1, the ord-th signal of the tile).
          const uint32_t need =
              hop ? (uint32_t)ti.ord : (fin ? (uint32_t)(p.R - 1) : (p.deterministic ? (uint32_t)ti.ord : 1u));
          const uint32_t have = __shfl_sync(0xffffffffu, lane == 0 ? ld_acquire_u32(ctr) : 0u, 0);
          int good = 1;
          if (have < need) {
            // Not yet: first publish this warp's own deferred partial (it
            // may be the one being waited for), then wait.
            publish(true);
            if (lane == 0) {
              good = wait_counter_geq(ctr, need, p.timeout_ns, abort_flag, gstatus) ? 1 : 0;
              if (!good && !*abort_flag && !*gstatus) record_error(p.status, FO_ERR_TIMEOUT, ti.r, ti.s, ti.c);
            }
          }
          if (lane == 0) fence_proxy_async_global();
          ok = __shfl_sync(0xffffffffu, good, 0) != 0;
          if (!ok) *abort_flag = 1;
        }
      }

      const size_t ncols = (size_t)p.n_cols;
      // Where a finisher reads the sum of the partials before its own: the
      // shard the others added into, or (ring) chunk c's rows of this rank's
      // receive buffer. The first partial of a tile has nothing to read.
      const float* sum_src = nullptr;
      if (EPI == EPI_RS && ti.ord > 0)
        sum_src = ring ? p.inbox[ti.r] + (size_t)ti.c * p.rows_per_chunk * ncols : p.shard[ti.c];
      if (EPI == EPI_RS && fin && last && p.completion == FO_COMPLETE_BF16) {
        // Finisher, bf16 output: 8 sub-tiles of 32 rows x 32 columns. The own
        // partial is staged fp32 in the warp's last buffer, the other R-1
        // partials' sum is added there with coalesced loads, and every pair
        // of sub-tiles is rounded once into 64-column bf16 rows, stored from
        // the other buffers. The sums of sub-tile j+1 are in flight while
        // sub-tile j is processed.
        static_assert(kEpiBufs >= 2, "the bf16 finisher needs two staging buffers per warp");
        constexpr int kSub = FO_BN / 32;
        const uint32_t addbuf = sEpi + (uint32_t)((e * kEpiBufs + kEpiBufs - 1) * kEpiBuf);
        float4 sum[2][8];
        uint32_t w[32];
        load_block32_coalesced(sum_src, row0, p.rows_per_chunk, n0, (int)ncols, ncols, lane, sum[0]);
        if (lane == 0) bulk_wait_read<0>();   // no store still reads a staging buffer
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
          uint32_t v[32];
          tmem_ld32(tbase + j * 32, v);
          if (j + 1 < kSub)
            load_block32_coalesced(sum_src, row0, p.rows_per_chunk, n0 + (j + 1) * 32, (int)ncols, ncols, lane,
                                   sum[(j + 1) & 1]);
          tmem_ld_wait();
          reg_fence(v);
          if (j == kSub - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
              else mbar_arrive(tempty_bar(acc));
            }
          }
          if (!ok) continue;
          stage_row_sw128(addbuf, lane, v);
          __syncwarp();
          add_block32_sw128(addbuf, lane, sum[j & 1]);
          __syncwarp();
          float f[32];
          read_row_sw128(addbuf, lane, f);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[(j & 1) * 16 + i] = *reinterpret_cast<uint32_t*>(&h);
          }
          if (j & 1) {
            const uint32_t buf = sEpi + (uint32_t)((e * kEpiBufs + (j >> 1) % (kEpiBufs - 1)) * kEpiBuf);
            if (lane == 0) bulk_wait_read<kEpiBufs - 2>();
            __syncwarp();
            stage_row_sw128(buf, lane, w);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&p.tmF[ti.c], buf, n0 + (j - 1) * 32, row0);
              bulk_commit();
            }
          }
        }
        if (ok && lane == 0) atomicExch(ctr, 0u);   // every partial is in: ready for the next call
      } else if (EPI == EPI_RS && fin) {
        // Finisher, all-reduce: 8 sub-tiles of 32 rows x 32 fp32 columns;
        // own partial + the other R-1 partials' sum, stored to the same rows
        // of every rank's full output (the all-gather half).
        // Ring hop, fp32: own partial + the running sum from the receive
        // buffer, forwarded into the next rank's receive buffer, or (last
        // hop) stored to the owner's output.
        // The own partial is staged row-per-lane (as it comes out of TMEM)
        // and the sum is added there with coalesced loads. The sums of
        // sub-tile j+1 are in flight while sub-tile j is processed.
        constexpr int kSub = FO_BN / 32;
        float4 sum[2][8];
        load_block32_coalesced(sum_src, row0, p.rows_per_chunk, n0, (int)ncols, ncols, lane, sum[0]);
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
          uint32_t v[32];
          tmem_ld32(tbase + j * 32, v);
          if (j + 1 < kSub)
            load_block32_coalesced(sum_src, row0, p.rows_per_chunk, n0 + (j + 1) * 32, (int)ncols, ncols, lane,
                                   sum[(j + 1) & 1]);
          tmem_ld_wait();
          reg_fence(v);
          if (j == kSub - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
              else mbar_arrive(tempty_bar(acc));
            }
          }
          if (!ok) continue;
          const uint32_t buf = sEpi + (uint32_t)((e * kEpiBufs + (j % kEpiBufs)) * kEpiBuf);
          if (lane == 0) bulk_wait_read<kEpiBufs - 1>();
          __syncwarp();
          stage_row_sw128(buf, lane, v);
          __syncwarp();
          add_block32_sw128(buf, lane, sum[j & 1]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (!ring)
              for (int qq = 0; qq < p.R; ++qq) tma_store_3d(&p.tmAR[qq], buf, n0 + j * 32, row0, ti.c);
            else if (last)
              tma_store_2d(&p.tmD[ti.c], buf, n0 + j * 32, row0);
            else
              tma_store_3d(&p.tmAR[(ti.r + 1) % p.R], buf, n0 + j * 32, row0, ti.c);
            bulk_commit();
          }
        }
        if (ok && last && lane == 0) atomicExch(ctr, 0u);   // every partial is in: ready for the next call
        if (ok && !last) {
          // Ring: the forward is in the next rank's buffer once its stores
          // are performed. Like a reduce tile's partial, it is released
          // after the next tile's stores are issued (or before this warp
          // blocks), so the warp does not wait for its own latest writes.
          publish(false);
          pend_ctr = ctr;
          pend_skip = false;
          if (in_split) publish(true);
        }
      } else if constexpr (EPI == EPI_AG) {
        // 4 sub-tiles of 32 rows x 64 bf16 columns.
#pragma unroll 1
        for (int j = 0; j < FO_BN / 64; ++j) {
          uint32_t v0[32], v1[32], w[32];
          tmem_ld32(tbase + j * 64, v0);
          tmem_ld32(tbase + j * 64 + 32, v1);
          tmem_ld_wait();
          reg_fence(v0);
          reg_fence(v1);
          if (j == FO_BN / 64 - 1) {
            // The accumulator may be refilled once every epilogue warp (of
            // both CTAs, for a pair) has read its quarter.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
              else mbar_arrive(tempty_bar(acc));
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
            __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
            w[i] = *reinterpret_cast<uint32_t*>(&h0);
            w[16 + i] = *reinterpret_cast<uint32_t*>(&h1);
          }
          // Stores go out in batches of kEpiBufs sub-tiles with one proxy
          // fence each, as in the reduce epilogue below.
          constexpr int kB = kEpiBufs;
          const uint32_t buf = sEpi + (uint32_t)((e * kEpiBufs + (j % kB)) * kEpiBuf);
          if (j % kB == 0) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
          stage_row_sw128(buf, lane, w);
          if (j % kB == kB - 1 || j == FO_BN / 64 - 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              for (int jj = j - (j % kB); jj <= j; ++jj) {
                const uint32_t bb = sEpi + (uint32_t)((e * kEpiBufs + (jj % kB)) * kEpiBuf);
                // Y is written once and never read here: its lines leave L2 first.
                const uint64_t pol = l2_policy_evict_first();
                if (p.a2a) tma_store_3d_hint(&p.tmD[ti.c], bb, n0 + jj * 64, row0, ti.r, pol);
                else tma_store_3d_hint(&p.tmD[ti.r], bb, n0 + jj * 64, row0, ti.c, pol);
                bulk_commit();
              }
            }
          }
        }
      } else {
        // 8 sub-tiles of 32 rows x 32 fp32 columns. The TMEM load of sub-tile
        // j+1 is in flight while sub-tile j is staged and sent.
        constexpr int kSub = FO_BN / 32;
        uint32_t v[2][32];
        tmem_ld32(tbase, v[0]);
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
          tmem_ld_wait();
          reg_fence(v[j & 1]);
          if (j + 1 < kSub) {
            tmem_ld32(tbase + (j + 1) * 32, v[(j + 1) & 1]);
          } else {
            // The accumulator may be refilled once every epilogue warp (of
            // both CTAs, for a pair) has read its quarter.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (PAIR) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
              else mbar_arrive(tempty_bar(acc));
            }
          }
          if (!ok) continue;
          // Sub-tiles go out kEpiBufs at a time: stage a batch (once the
          // previous batch's stores have read the buffers), one proxy fence,
          // then one TMA op per sub-tile. On the 8192 x 4096 x 1792 R = 8
          // reduce-scatter this ran 2.8% faster than one fence and op per
          // sub-tile with one buffer still in flight (1.7% on the DP
          // gradient); removing the fences alone gained nothing.
          constexpr int kB = kEpiBufs;
          const uint32_t buf = sEpi + (uint32_t)((e * kEpiBufs + (j % kB)) * kEpiBuf);
          if (j % kB == 0) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
          }
          stage_row_sw128(buf, lane, v[j & 1]);
          if (j % kB == kB - 1 || j == kSub - 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int jj = j - (j % kB); jj <= j; ++jj) {
                const uint32_t bb = sEpi + (uint32_t)((e * kEpiBufs + (jj % kB)) * kEpiBuf);
                if constexpr (EPI == EPI_PARTIAL) {
                  tma_store_3d(&p.tmD[ti.r], bb, n0 + jj * 32, row0, ti.c);
                } else {
                  if (ti.ord != 0) tma_reduce_add_2d(&p.tmD[ti.c], bb, n0 + jj * 32, row0);
                  else if (ring && !last) tma_store_3d(&p.tmAR[(ti.r + 1) % p.R], bb, n0 + jj * 32, row0, ti.c);
                  else tma_store_2d(&p.tmD[ti.c], bb, n0 + jj * 32, row0);
                }
                bulk_commit();
              }
            }
          }
        }
        if constexpr (EPI == EPI_RS) {
          if (ok) {
            // Publish the previous tile's partial (its 8 bulk groups are
            // older than this tile's 8) and keep this one pending, so the
            // warp never stalls on its own latest writes.
            publish(false);
            pend_ctr = ctr;
            pend_skip = p.fault_inject == FO_INJECT_SKIP_SIGNAL && ti.c == 0 && mt128 == 0 && ti.nt == 0 &&
                        q == 0 && ti.ord == 0;
            // With a finisher waiting for every other partial of the tile,
            // publishing late would stall it: publish this one now.
            if (p.completion != FO_COMPLETE_NONE || in_split) publish(true);
          }
        }
      }
    }
    if constexpr (EPI == EPI_RS) {
      const int aborted = __shfl_sync(0xffffffffu, lane == 0 ? (int)*abort_flag : 0, 0);
      if (!aborted) publish(true);
    }
    if (lane == 0) bulk_wait<0>();
    if (trace && lane == 0) trace[2 + e] = globaltimer();
    __syncwarp();
  }

  if constexpr (MOV) {
    if (warp >= 2 + kEpiWarps) {
      // ---------------------------------------------------------- movers
      // Shard pieces into the gather buffers, 128-bit copies. Piece (src,
      // pc) always belongs to the same CTA, so along the ring each copy reads
      // what this CTA's movers wrote one step earlier (same threads, same
      // bytes). Copy transport: rank r's piece of shard src = table[r][s]
      // comes from X_r at step 0 and from G_{r-1} after; a release flag per
      // piece tells the GEMM it is there. Peer-read transport: G_r[src] is a
      // side output copied straight from X_src. Movers never wait.
      const int mtid = threadIdx.x - 32 * (2 + kEpiWarps);
      constexpr int kMovThreads = 32 * kMoverWarps;
      const int R = p.R;
      const size_t rb = (size_t)p.row_bytes;
      const int rpc = p.rows_per_chunk;
      for (int s = 0; s < R; ++s) {
        for (int r = 0; r < R; ++r) {
          const int src = p.table[r][s];
          for (int pc = 0; pc < p.pieces; ++pc) {
            if ((src * p.pieces + pc) % (int)gridDim.x != (int)blockIdx.x) continue;
            const int rows = min(kPieceRows, rpc - pc * kPieceRows);
            const size_t shard_off = ((size_t)src * rpc + (size_t)pc * kPieceRows) * rb;
            const uint8_t* from = (p.ag_copy && s > 0)
                                      ? static_cast<const uint8_t*>(p.gdst[(r + R - 1) % R]) + shard_off
                                      : static_cast<const uint8_t*>(p.xsrc[src]) + (size_t)pc * kPieceRows * rb;
            uint8_t* to = static_cast<uint8_t*>(p.gdst[r]) + shard_off;
            copy16(from, to, (size_t)rows * rb / 16, mtid, kMovThreads);
            if (p.ag_copy) {
              __threadfence();
              named_bar_sync(1, kMovThreads);
              const bool skip = p.fault_inject == FO_INJECT_SKIP_SIGNAL && R > 1 && r == 1 && s == 1 && pc == 0;
              if (mtid == 0 && !skip) st_release_u32(&p.flags[((size_t)r * R + src) * p.pieces + pc], epoch0 + 1u);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();   // neither CTA leaves while the pair still uses its memory
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
  if (trace && threadIdx.x == 0) trace[6] = globaltimer();
  if constexpr (MOV) {
    // The last CTA of the launch advances the flag epoch for the next call.
    if (threadIdx.x == 0 && p.ag_copy) {
      __threadfence();
      const uint32_t done = atomicAdd(p.epoch + 1, 1u);
      if (done == gridDim.x - 1) {
        atomicExch(p.epoch + 1, 0u);
        __threadfence();
        atomicAdd(p.epoch, 1u);
      }
    }
  }
}

}  // namespace fo

// Launchers, one per compiled variant (defined in the fo_kern_*.cu files).
enum fo_variant {
  FO_V_RS_BF16_KN = 0,
  FO_V_RS_BF16_NK,
  FO_V_RS_TF32_NK,
  FO_V_DP_BF16,
  FO_V_AG_BF16_KN,
  FO_V_AG_BF16_NK,
  FO_V_PART_BF16_KN,
  FO_V_PART_BF16_NK,
  FO_V_PART_TF32_NK,
  FO_V_PART_DP,
  FO_V_AG_BF16_KN_MOV,
  FO_V_AG_BF16_NK_MOV,
  FO_V_AG_BF16_KN_GST,
  FO_V_AG_BF16_NK_GST,
  FO_V_RS_BF16_KN_SK,   // GEMM-RS with few k-blocks a task (CTA pairs only)
  FO_V_COUNT
};

// Launch `variant` with single-CTA tiles (pair = false) or CTA-pair tiles;
// `grid` counts CTAs (even for pairs).
cudaError_t fo_launch_variant(int variant, bool pair, const fo::FoParams& p, int grid, cudaStream_t stream);
// Largest grid (CTAs) of this variant that can be resident at once.
cudaError_t fo_max_resident_ctas(int variant, bool pair, int* ctas);
