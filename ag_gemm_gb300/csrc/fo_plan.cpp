// Host-side schedule builder and validator (fo_plan and its accessors).
//
// The schedule follows the pages about FlashOverlap (arXiv 2604.24013):
//  * a collective becomes a set of directed P2P chunk transfers (euno.news,
//    "Methodology" item 1);
//  * Flash-RS computes the chunk that stays on the rank last (gist.science,
//    "Technical Summary" section 2, Flash-Reduce-Scatter);
//  * Flash-AG computes the rank's own shard first and then the shards that
//    arrive along a ring (same section, Flash-All-Gather);
//  * the transfers and compute fragments form a dependency graph in which no
//    sub-task waits for a last piece of data (euno.news, "Methodology" 3).
// The order of the chunks in between is this library's reading: RS follows
// the ring reduce-scatter order, chunk (r - 1 - s) mod R at step s, so that
// every owner receives exactly one partial per step; AG consumes the shard of
// rank (r - s) mod R, which its ring predecessor forwarded one step earlier.
// Under the ring RS algorithm the same order makes rank r's chunk at step s
// the one rank r-1 handled at step s-1, so the running sum can be forwarded.
// Flash All-to-All (gist.science, "Technical Summary" section 2, named for
// Ulysses parallelism) takes the RS table too: rank r computes the column
// block of rank (r - 1 - s) mod R at step s and sends it straight there, the
// block that stays last; its transfers and edges are those of the direct RS.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "fo_internal.h"

namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int fo_tail_split_tiles(int64_t total, int units) {
  if (units <= 0 || total <= units) return 0;
  const int64_t waves = total / units, rem = total % units;
  if (rem == 0) return 0;
  const double idle = (double)(units - rem) / ((double)units * (double)(waves + 1));
  if (idle <= 0.02) return 0;
  // Two whole waves plus the partial one where there are that many, so that
  // each unit's share (about two tiles) ends in a whole tile, whose math
  // hides the finishing part's extra epilogue work.
  return (int)(waves >= 2 ? 2 * units + rem : total);
}

// Host logging to stderr when the environment has FO_LOG=1 (read once).
bool fo_log_enabled() {
  static const bool on = [] {
    const char* v = getenv("FO_LOG");
    return v && v[0] == '1' && v[1] == 0;
  }();
  return on;
}

namespace {
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool is_perm(const int32_t* v, int n, int stride) {
  bool seen[FO_MAX_R] = {false};
  for (int i = 0; i < n; ++i) {
    int x = v[i * stride];
    if (x < 0 || x >= n || seen[x]) return false;
    seen[x] = true;
  }
  return true;
}

void build_table(fo_plan_s* p) {
  const int R = p->R;
  const bool ag = p->d.op == FO_OP_AG_GEMM;
  for (int r = 0; r < R; ++r)
    for (int s = 0; s < R; ++s) {
      if (p->d.sched == FO_SCHED_SLICED) p->table[r][s] = s;
      else if (ag) p->table[r][s] = ((r - s) % R + R) % R;
      else p->table[r][s] = ((r - 1 - s) % R + 2 * R) % R;
    }
  // The kernel's task order.
  int skew = p->d.interleave;
  if (skew == FO_INTERLEAVE_AUTO) {
    // Ring reduce-scatter and ring-forwarded all-gather: a chain's hops run
    // a whole step apart, so no hop waits for the one before.
    if (p->ring || (ag && p->d.ag_transport == FO_AG_COPY)) skew = FO_INTERLEAVE_LOCKSTEP;
    else skew = (ag || p->d.op == FO_OP_DP_GRAD_RS || p->d.op == FO_OP_GEMM_A2A) ? FO_INTERLEAVE_RANK_MAJOR
                                                                                  : FO_INTERLEAVE_SKEWED_PAIRS;
  }
  int n = 0;
  if (skew == FO_INTERLEAVE_RANK_MAJOR) {
    for (int r = 0; r < R; ++r)
      for (int s = 0; s < R; ++s) {
        p->task_r[n] = r;
        p->task_s[n] = s;
        ++n;
      }
  } else if (skew == FO_INTERLEAVE_SKEWED_PAIRS) {
    // Slots t and t + 1 together: rank r runs its steps t + r and t + 1 + r
    // back to back (ranks in ascending order, as in a single slot).
    for (int t = -(R - 1); t <= R - 1; t += 2)
      for (int r = 0; r < R; ++r)
        for (int dt = 0; dt < 2 && t + dt <= R - 1; ++dt) {
          const int s = t + dt + r;
          if (s < 0 || s >= R) continue;
          p->task_r[n] = r;
          p->task_s[n] = s;
          ++n;
        }
  } else if (skew == FO_INTERLEAVE_SKEWED) {
    // Slot t = s - r (rank r runs r steps behind rank 0); inside a slot by
    // ascending step, so every shard receives its partials in step order.
    for (int t = -(R - 1); t <= R - 1; ++t)
      for (int s = 0; s < R; ++s) {
        const int r = s - t;
        if (r < 0 || r >= R) continue;
        p->task_r[n] = r;
        p->task_s[n] = s;
        ++n;
      }
  } else {
    // Lockstep; RS/DP ranks alternate direction from step to step.
    int order[FO_MAX_R];
    for (int i = 0; i < R; ++i) order[i] = i;
    for (int s = 0; s < R; ++s) {
      for (int i = 0; i < R; ++i) {
        p->task_r[n] = order[i];
        p->task_s[n] = s;
        ++n;
      }
      if (!ag) {
        int next[FO_MAX_R];
        for (int i = 0; i < R; ++i) next[i] = (order[R - 1 - i] + 1) % R;
        for (int i = 0; i < R; ++i) order[i] = next[i];
      }
    }
  }
  // Contribution order of every (r, s) into its chunk, in the kernel's order.
  int seen[FO_MAX_R] = {0};
  for (int i = 0; i < R * R; ++i) {
    const int r = p->task_r[i], s = p->task_s[i];
    p->ord[r][s] = seen[p->table[r][s]]++;
  }
}

void build_transfers_and_edges(fo_plan_s* p) {
  const int R = p->R;
  p->transfers.clear();
  p->edges.clear();
  for (int r = 0; r < R; ++r)
    for (int s = 0; s + 1 < R; ++s) p->edges.push_back({r, s, r, s + 1});
  if (p->d.op == FO_OP_AG_GEMM || p->ring) {
    // Ring: after using shard table[r][s] (AG), or adding its partial to the
    // running sum of chunk table[r][s] (ring RS), rank r forwards it to r+1,
    // which consumes it at step s+1. Nothing is forwarded after the last step.
    for (int s = 0; s + 1 < R; ++s)
      for (int r = 0; r < R; ++r) p->transfers.push_back({r, (r + 1) % R, p->table[r][s], s});
    for (const fo_transfer& t : p->transfers) p->edges.push_back({t.src, t.step, t.dst, t.step + 1});
  } else {
    // Direct RS: a non-own partial goes to its owner, whose own-chunk task
    // (the one that finalises its shard) must come after it.
    for (int s = 0; s < R; ++s)
      for (int r = 0; r < R; ++r) {
        int c = p->table[r][s];
        if (c != r) p->transfers.push_back({r, c, c, s});
      }
    for (const fo_transfer& t : p->transfers) {
      int own = 0;
      for (int s = 0; s < R; ++s)
        if (p->table[t.dst][s] == t.dst) own = s;
      p->edges.push_back({t.src, t.step, t.dst, own});
    }
  }
  if (p->d.fault_inject == FO_INJECT_DROP_TRANSFER && !p->transfers.empty()) p->transfers.pop_back();
}

// All-reduce = reduce-scatter then all-gather: once shard c is complete its
// owner sends it to every other rank (listed as step R, after the RS steps).
void add_allgather_half(fo_plan_s* p) {
  const int R = p->R;
  for (int c = 0; c < R; ++c)
    for (int q = 0; q < R; ++q)
      if (q != c) p->transfers.push_back({c, q, c, R});
}

bool dag_acyclic(const fo_plan_s* p) {
  const int R = p->R, n = R * R;
  std::vector<int> indeg(n, 0);
  std::vector<std::vector<int>> adj(n);
  for (const fo_edge& e : p->edges) {
    int a = e.ra * R + e.sa, b = e.rb * R + e.sb;
    if (a == b) continue;  // an edge from a task to itself orders nothing
    adj[a].push_back(b);
    indeg[b]++;
  }
  std::vector<int> stack;
  for (int i = 0; i < n; ++i)
    if (!indeg[i]) stack.push_back(i);
  int seen = 0;
  while (!stack.empty()) {
    int a = stack.back();
    stack.pop_back();
    ++seen;
    for (int b : adj[a])
      if (--indeg[b] == 0) stack.push_back(b);
  }
  return seen == n;
}

fo_status validate(const fo_plan_s* p) {
  const int R = p->R;
  const bool ag = p->d.op == FO_OP_AG_GEMM;
  const bool adaptive = p->d.sched == FO_SCHED_RANK_ADAPTIVE;
  for (int r = 0; r < R; ++r)
    if (!is_perm(&p->table[r][0], R, 1)) return FO_ERR_PLAN_INVARIANT;          // (i)
  if ((int64_t)p->transfers.size() != (int64_t)R * (R - 1)) return FO_ERR_PLAN_INVARIANT;  // (v)
  if (!dag_acyclic(p)) return FO_ERR_PLAN_INVARIANT;                             // (iv)
  if (!adaptive) return FO_OK;
  for (int r = 0; r < R; ++r) {                                                  // (ii)
    if (ag ? p->table[r][0] != r : p->table[r][R - 1] != r) return FO_ERR_PLAN_INVARIANT;
  }
  for (const fo_transfer& t : p->transfers)
    if (t.step >= R - 1) return FO_ERR_PLAN_INVARIANT;                           // no tail send
  for (int s = 0; s < R; ++s)
    if (!is_perm(&p->table[0][s], R, FO_MAX_R)) return FO_ERR_PLAN_INVARIANT;   // (iii)
  if (p->ring) {
    // Ring RS: every forward carries the chunk its sender handled at that
    // step to the next rank, which handles the same chunk one step later;
    // every rank receives R-1 forwards, all from its ring predecessor.
    int recv[FO_MAX_R] = {0};
    for (const fo_transfer& t : p->transfers) {
      if (t.dst != (t.src + 1) % R || t.step < 0 || t.step + 1 >= R) return FO_ERR_PLAN_INVARIANT;
      if (p->table[t.src][t.step] != t.chunk || p->table[t.dst][t.step + 1] != t.chunk)
        return FO_ERR_PLAN_INVARIANT;
      ++recv[t.dst];
    }
    for (int r = 0; r < R; ++r)
      if (recv[r] != R - 1) return FO_ERR_PLAN_INVARIANT;
    // The kernel adds each chunk's partials in the order it runs them: that
    // order must be the chain's (hop s = step s).
    for (int r = 0; r < R; ++r)
      for (int s = 0; s < R; ++s)
        if (p->ord[r][s] != s) return FO_ERR_UNSUPPORTED;
  } else if (ag) {
    // Every shard a rank consumes after step 0 arrives by a transfer of that
    // shard to that rank at an earlier step.
    for (int r = 0; r < R; ++r)
      for (int s = 1; s < R; ++s) {
        bool ok = false;
        for (const fo_transfer& t : p->transfers)
          ok |= t.dst == r && t.chunk == p->table[r][s] && t.step < s;
        if (!ok) return FO_ERR_PLAN_INVARIANT;
      }
  } else {
    // Every partial for owner c is sent before c's own-chunk task, and each
    // owner receives exactly R-1 partials, one per other rank.
    for (int c = 0; c < R; ++c) {
      int n = 0;
      for (const fo_transfer& t : p->transfers)
        if (t.dst == c) {
          ++n;
          if (t.step >= R - 1 || t.src == c) return FO_ERR_PLAN_INVARIANT;
        }
      if (n != R - 1) return FO_ERR_PLAN_INVARIANT;
    }
  }
  return FO_OK;
}

}  // namespace

extern "C" {

fo_status fo_plan(const fo_plan_desc* d, fo_plan_t* out) {
  if (!d || !out) return FO_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->op < FO_OP_AG_GEMM || d->op > FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
  if (d->R < 1 || d->R > FO_MAX_R) return FO_ERR_INVALID_ARG;
  if (d->sched != FO_SCHED_RANK_ADAPTIVE && d->sched != FO_SCHED_SLICED) return FO_ERR_INVALID_ARG;
  if (d->ag_transport != FO_AG_PEER_READ && d->ag_transport != FO_AG_COPY) return FO_ERR_INVALID_ARG;
  if (d->w_layout != FO_W_KN && d->w_layout != FO_W_NK) return FO_ERR_INVALID_ARG;
  if (d->fault_inject < FO_INJECT_NONE || d->fault_inject > FO_INJECT_DELAY_FIRST_TASK) return FO_ERR_INVALID_ARG;
  if (d->inject_delay_us < 0 || d->inject_delay_us > 1000000) return FO_ERR_INVALID_ARG;
  if (d->inject_delay_us && d->fault_inject != FO_INJECT_DELAY_FIRST_TASK) return FO_ERR_INVALID_ARG;
  if (d->trace != 0 && d->trace != 1) return FO_ERR_INVALID_ARG;
  if (d->tail_split < FO_TAIL_SPLIT_AUTO || d->tail_split > FO_TAIL_SPLIT_ON) return FO_ERR_INVALID_ARG;
  if (d->tile_config != FO_TILE_AUTO && d->tile_config != FO_TILE_SINGLE) return FO_ERR_INVALID_ARG;
  if (d->interleave < FO_INTERLEAVE_AUTO || d->interleave > FO_INTERLEAVE_SKEWED_PAIRS) return FO_ERR_INVALID_ARG;
  if (d->rs_algo != FO_RS_DIRECT && d->rs_algo != FO_RS_RING) return FO_ERR_INVALID_ARG;
  if (d->reserved[0]) return FO_ERR_INVALID_ARG;
  if (d->rs_algo == FO_RS_RING) {
    // The ring forwards a running sum, which needs the rank-adaptive order
    // (rank r's chunk at step s is r-1's at step s-1) and a kernel order that
    // runs every chunk's hops in step order.
    if (d->op == FO_OP_AG_GEMM || d->op == FO_OP_GEMM_A2A) return FO_ERR_INVALID_ARG;
    if (d->op == FO_OP_GEMM_AR || d->sched != FO_SCHED_RANK_ADAPTIVE) return FO_ERR_UNSUPPORTED;
    if (d->interleave == FO_INTERLEAVE_RANK_MAJOR) return FO_ERR_UNSUPPORTED;
  }
  if (d->M <= 0 || d->N <= 0 || d->K <= 0) return FO_ERR_SHAPE;
  const int R = d->R;
  const int64_t M = d->M, N = d->N, K = d->K;
  if (M % R) return FO_ERR_SHAPE;
  if (M / R > (int64_t)1 << 30 || N > (int64_t)1 << 30 || K > (int64_t)1 << 30) return FO_ERR_SHAPE;

  int eb = 2;
  switch (d->op) {
    case FO_OP_GEMM_RS:
    case FO_OP_GEMM_AR:
      if (K % R) return FO_ERR_SHAPE;
      if (d->out_dtype != FO_F32 && !(d->op == FO_OP_GEMM_RS && d->out_dtype == FO_BF16)) return FO_ERR_DTYPE;
      if (d->in_dtype == FO_F32) {
        eb = 4;   // fp32 operands feed the tf32 MMA (a [K x N] W is transposed first)
      } else if (d->in_dtype != FO_BF16) {
        return FO_ERR_DTYPE;
      }
      if (((K / R) * eb) % 16) return FO_ERR_ALIGN;   // rows of X_r (and of W_r if NK)
      if ((N * eb) % 16) return FO_ERR_ALIGN;         // rows of W_r (KN)
      if ((N * 4) % 16) return FO_ERR_ALIGN;          // rows of Y
      if (d->out_dtype == FO_BF16 && (N * 2) % 16) return FO_ERR_ALIGN;   // rows of a bf16 Y
      break;
    case FO_OP_AG_GEMM:
      if (N % R) return FO_ERR_SHAPE;
      if (d->in_dtype != FO_BF16 || d->out_dtype != FO_BF16) return FO_ERR_DTYPE;
      if (d->sched != FO_SCHED_RANK_ADAPTIVE) return FO_ERR_UNSUPPORTED;
      if ((K * 2) % 16 || ((N / R) * 2) % 16) return FO_ERR_ALIGN;
      break;
    case FO_OP_GEMM_A2A:
      // Column block c of W_r starts at column c*N/R: a TMA coordinate along
      // the contiguous dimension of a [K x N] weight, so it falls on a
      // 16-byte boundary only when N/R bf16 values fill whole 16 bytes.
      if (N % R) return FO_ERR_SHAPE;
      if (d->in_dtype != FO_BF16 || d->out_dtype != FO_BF16) return FO_ERR_DTYPE;
      if (d->ag_transport != FO_AG_PEER_READ) return FO_ERR_INVALID_ARG;
      if ((K * 2) % 16 || ((N / R) * 2) % 16) return FO_ERR_ALIGN;
      break;
    case FO_OP_DP_GRAD_RS:
      if (d->in_dtype != FO_BF16) return FO_ERR_DTYPE;
      if (d->out_dtype != FO_F32 && d->out_dtype != FO_BF16) return FO_ERR_DTYPE;
      if (d->w_layout != FO_W_KN) return FO_ERR_INVALID_ARG;
      // A chunk starts at column c*M/R of X_r: a TMA coordinate along the
      // contiguous dimension, so it must fall on a 16-byte boundary.
      if (((M / R) * 2) % 16) return FO_ERR_ALIGN;
      if ((M * 2) % 16 || (N * 2) % 16) return FO_ERR_ALIGN;
      if ((N * 4) % 16) return FO_ERR_ALIGN;
      break;
  }

  fo_plan_s* p = new (std::nothrow) fo_plan_s();
  if (!p) return FO_ERR_INVALID_ARG;
  p->d = *d;
  if (!p->d.timeout_ns) p->d.timeout_ns = 1000000000ull;
  p->R = R;
  p->ring = d->rs_algo == FO_RS_RING;
  p->elem_bytes = eb;
  p->rows_per_chunk = M / R;
  switch (d->op) {
    case FO_OP_GEMM_RS:
    case FO_OP_GEMM_AR: p->k_red = K / R; p->n_out = N; break;
    case FO_OP_AG_GEMM:
    case FO_OP_GEMM_A2A: p->k_red = K; p->n_out = N / R; break;
    default: p->k_red = K; p->n_out = N; break;
  }
  // AUTO: CTA-pair tiles for bf16 unless a shard holds 128 rows or fewer,
  // where a 256-row pair tile would be mostly padding.
  p->pair = eb == 2 && d->tile_config == FO_TILE_AUTO && M / R > FO_BM;
  p->tiles_m = (int)cdiv(p->rows_per_chunk, p->pair ? 2 * FO_BM : FO_BM);
  p->ctr_tiles_m = 2 * (int)cdiv(p->rows_per_chunk, 2 * FO_BM);
  p->pieces = (int)cdiv(p->rows_per_chunk, 32);
  p->tiles_n = (int)cdiv(p->n_out, FO_BN);
  p->num_kb = (int)cdiv(p->k_red * eb, FO_BK_BYTES);
  if ((int64_t)R * R * p->tiles_m * p->tiles_n > ((int64_t)1 << 31) - 1) {
    delete p;
    return FO_ERR_SHAPE;
  }
  build_table(p);
  build_transfers_and_edges(p);
  fo_status st = validate(p);
  if (st != FO_OK) {
    delete p;
    return st;
  }
  if (d->op == FO_OP_GEMM_AR) add_allgather_half(p);
  size_t off = align_up(sizeof(fo_ws_header), 256);
  p->ws_counters_off = off;
  p->ws_flags_off = off;
  if (d->op == FO_OP_AG_GEMM) {
    off += align_up((size_t)R * R * p->pieces * sizeof(uint32_t), 256);
  } else if (d->op != FO_OP_GEMM_A2A) {   // the all-to-all's blocks are disjoint: no counters
    off += align_up((size_t)R * p->ctr_tiles_m * p->tiles_n * 4 * sizeof(uint32_t), 256);
  }
  p->ws_shard_off = off;
  p->ws_shard_stride = 0;
  if (d->op != FO_OP_AG_GEMM && d->op != FO_OP_GEMM_A2A && d->out_dtype == FO_BF16 && !p->ring) {
    p->ws_shard_stride = align_up((size_t)p->rows_per_chunk * p->n_out * 4, 256);
    off += (size_t)R * p->ws_shard_stride;
  }
  // Ring RS: each rank's receive buffer holds one fp32 chunk per sender
  // step; a rank receives each chunk at most once per call, so a chunk-
  // indexed buffer of all M rows needs no reuse within a call.
  p->ws_ring_off = off;
  p->ws_ring_stride = 0;
  if (p->ring) {
    p->ws_ring_stride = align_up((size_t)p->rows_per_chunk * R * p->n_out * 4, 256);
    off += (size_t)R * p->ws_ring_stride;
  }
  // fp32 inputs with W as [K x N]: the tf32 MMA reads B K-major only, so
  // each call transposes W_r into this region first.
  p->ws_wt_off = off;
  p->ws_wt_stride = 0;
  if (eb == 4 && d->w_layout == FO_W_KN) {
    p->ws_wt_stride = align_up((size_t)p->k_red * p->n_out * 4, 256);
    off += (size_t)R * p->ws_wt_stride;
  }
  p->ws_trace_off = off;
  if (d->trace) off += align_up((size_t)FO_TRACE_MAX_CTAS * FO_TRACE_STAMPS * sizeof(uint64_t), 256);
  // Tail split, sized for a GB300's units (a launch on fewer or more units
  // uses it only when its split fits).
  p->ws_split_off = off;
  p->sk_cap = 0;
  {
    const int64_t tiles = (int64_t)R * R * p->tiles_m * p->tiles_n;
    const int units = p->pair ? FO_GB300_SMS / 2 : FO_GB300_SMS;
    const bool on = d->tail_split == FO_TAIL_SPLIT_ON ||
                    (d->tail_split == FO_TAIL_SPLIT_AUTO &&
                     (d->op == FO_OP_AG_GEMM || d->op == FO_OP_GEMM_A2A) && p->num_kb >= 32 &&
                     tiles >= 2 * (int64_t)units);
    if (on) p->sk_cap = fo_tail_split_tiles(tiles, units);
  }
  if (p->sk_cap) {
    off += align_up((size_t)p->sk_cap * (p->pair ? 2 * FO_BM : FO_BM) * FO_BN * 4, 256);
    p->ws_split_ctr_off = off;
    off += align_up((size_t)p->sk_cap * 8 * sizeof(uint32_t), 256);
  } else {
    p->ws_split_ctr_off = off;
  }
  p->ws_bytes = off;
  p->last_launches = 0;
  p->last_grid = 0;
  p->last_split_tiles = 0;
  p->param_cache = nullptr;
  if (fo_log_enabled()) {
    static const char* ops[] = {"ag_gemm", "gemm_rs", "dp_grad_rs", "gemm_ar", "gemm_a2a"};
    fprintf(stderr,
            "[flashoverlap] plan %s R=%d M=%lld N=%lld K=%lld %s tiles %dx%d of %s, %d k-blocks, %s%s, "
            "tail split for up to %d tiles, workspace %zu B\n",
            ops[d->op], R, (long long)M, (long long)N, (long long)K, eb == 4 ? "tf32" : "bf16", p->tiles_m,
            p->tiles_n, p->pair ? "256x256 (CTA pair)" : "128x256", p->num_kb,
            d->sched == FO_SCHED_SLICED ? "sliced" : "rank-adaptive", p->ring ? ", ring RS" : "", p->sk_cap,
            p->ws_bytes);
  }
  *out = p;
  return FO_OK;
}

void fo_plan_destroy(fo_plan_t p) {
  if (!p) return;
  free(p->param_cache);
  delete p;
}

fo_status fo_plan_table(fo_plan_t p, int32_t* table) {
  if (!p || !table) return FO_ERR_INVALID_ARG;
  for (int r = 0; r < p->R; ++r)
    for (int s = 0; s < p->R; ++s) table[r * p->R + s] = p->table[r][s];
  return FO_OK;
}

fo_status fo_plan_task_order(fo_plan_t p, int32_t* order) {
  if (!p || !order) return FO_ERR_INVALID_ARG;
  for (int i = 0; i < p->R * p->R; ++i) {
    order[2 * i] = p->task_r[i];
    order[2 * i + 1] = p->task_s[i];
  }
  return FO_OK;
}

fo_status fo_plan_transfers(fo_plan_t p, int32_t* out, int32_t cap, int32_t* n) {
  if (!p || !n || (cap > 0 && !out) || cap < 0) return FO_ERR_INVALID_ARG;
  *n = (int32_t)p->transfers.size();
  for (int i = 0; i < *n && i < cap; ++i) {
    const fo_transfer& t = p->transfers[i];
    out[4 * i + 0] = t.src;
    out[4 * i + 1] = t.dst;
    out[4 * i + 2] = t.chunk;
    out[4 * i + 3] = t.step;
  }
  return *n <= cap ? FO_OK : FO_ERR_INVALID_ARG;
}

fo_status fo_plan_edges(fo_plan_t p, int32_t* out, int32_t cap, int32_t* n) {
  if (!p || !n || (cap > 0 && !out) || cap < 0) return FO_ERR_INVALID_ARG;
  *n = (int32_t)p->edges.size();
  for (int i = 0; i < *n && i < cap; ++i) {
    const fo_edge& e = p->edges[i];
    out[4 * i + 0] = e.ra;
    out[4 * i + 1] = e.sa;
    out[4 * i + 2] = e.rb;
    out[4 * i + 3] = e.sb;
  }
  return *n <= cap ? FO_OK : FO_ERR_INVALID_ARG;
}

fo_status fo_workspace_size(fo_plan_t p, size_t* bytes) {
  if (!p || !bytes) return FO_ERR_INVALID_ARG;
  *bytes = p->ws_bytes;
  return FO_OK;
}

int32_t fo_plan_last_launches(fo_plan_t p) { return p ? p->last_launches : -1; }

int32_t fo_plan_last_split_tiles(fo_plan_t p) { return p ? p->last_split_tiles : -1; }

const char* fo_status_string(fo_status s) {
  switch (s) {
    case FO_OK: return "ok";
    case FO_ERR_INVALID_ARG: return "invalid argument";
    case FO_ERR_SHAPE: return "unsupported or inconsistent shape";
    case FO_ERR_DTYPE: return "unsupported dtype combination";
    case FO_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
    case FO_ERR_UNSUPPORTED: return "option or device not supported";
    case FO_ERR_CUDA: return "CUDA call failed";
    case FO_ERR_TIMEOUT: return "device-side wait timed out";
    case FO_ERR_PLAN_INVARIANT: return "schedule failed a validity check";
    case FO_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the static no-alloc buffer holds";
  }
  return "unknown status";
}

int32_t fo_version(void) { return 0x000100; }

}  // extern "C"
