/*
 * flashoverlap.h - C ABI of libflashoverlap.so: FlashOverlap's partitioned
 * GEMM fused with a decomposed reduce-scatter or all-gather, with R virtual
 * ranks held as separate buffers on one GB300 (sm_103a).
 *
 * The method (arXiv 2604.24013, as described on the pages cited below):
 *   - a collective (reduce-scatter, all-gather) is replaced by directed
 *     point-to-point chunk transfers (euno.news summary, "Methodology" item 1;
 *     gist.science "Technical Summary" section 2);
 *   - the GEMM is split into sub-tasks over exactly the slices that are
 *     communicated (euno.news, "Methodology" item 2);
 *   - the sub-tasks run in a rank-adaptive order: Flash-RS computes the slice
 *     that stays on the rank last, Flash-AG computes the rank's own slice
 *     first and then the slices received along a ring (gist.science,
 *     "Technical Summary" section 2, Flash-Reduce-Scatter / Flash-All-Gather);
 *   - a dependency graph of transfers and compute fragments is scheduled so
 *     that no sub-task waits for a last piece of data (euno.news,
 *     "Methodology" item 3); a synchronisation mechanism keeps the data
 *     consistent (shd-paper.top, 方法详解 "key design" paragraph, item 3).
 *
 * On one GPU a "rank" is a set of buffers and a "P2P transfer" is either an
 * fp32 accumulate of a partial tile into the owning rank's shard (RS) or an
 * in-kernel read of another rank's buffer (AG). No NCCL, no second GPU.
 *
 * Conventions for every call below:
 *   - Ownership: the caller owns every device buffer (inputs, outputs, the
 *     workspace) and the stream. The library owns the plan (host memory only;
 *     a plan holds no device memory) and frees it in fo_plan_destroy.
 *   - Pointer arrays (X, W, Y, ...) are HOST arrays of R DEVICE pointers, one
 *     per virtual rank; each device pointer must be 16-byte aligned.
 *   - All matrices are dense row-major with no padding between rows.
 *   - Launching calls are asynchronous on `stream` and return after launch.
 *   - Errors found on the host return at once and launch nothing. Errors
 *     found on the device (a bounded wait that ran out) are recorded in the
 *     workspace and reported by fo_status_query.
 *   - No call aborts the process or lets a C++ exception escape.
 *   - One call per workspace may be in flight at a time.
 */
#ifndef FLASHOVERLAP_H
#define FLASHOVERLAP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* fo_stream_t;

typedef enum {
  FO_OK = 0,
  FO_ERR_INVALID_ARG = 1,     /* NULL pointer, bad enum value, R out of range */
  FO_ERR_SHAPE = 2,           /* a size is not positive or not divisible by R */
  FO_ERR_DTYPE = 3,           /* dtype combination not offered for this op */
  FO_ERR_ALIGN = 4,           /* pointer or row stride not 16-byte aligned */
  FO_ERR_UNSUPPORTED = 5,     /* option not built, or device is not sm_103 */
  FO_ERR_CUDA = 6,            /* a CUDA runtime/driver call failed */
  FO_ERR_TIMEOUT = 7,         /* a device-side bounded wait ran out */
  FO_ERR_PLAN_INVARIANT = 8,  /* the schedule failed a validity check */
  FO_ERR_SCRATCH_LIMIT = 9    /* fo_gemm_rs_noalloc: problem needs more scratch
                                 than its static buffer holds */
} fo_status;

typedef enum {
  FO_OP_AG_GEMM = 0,          /* Y_r = AllGather(X) . W_r           */
  FO_OP_GEMM_RS = 1,          /* Y   = ReduceScatter(X_r . W_r)     */
  FO_OP_DP_GRAD_RS = 2,       /* dW  = ReduceScatter(X_r^T . dY_r)  */
  FO_OP_GEMM_AR = 3,          /* Y_r = AllReduce(X_q . W_q) = RS then AG */
  FO_OP_GEMM_A2A = 4          /* Y_c = AllToAll(X_r . W_r): block c of every rank */
} fo_op;

typedef enum { FO_BF16 = 0, FO_F32 = 1 } fo_dtype;

/* Per-rank order of the chunk tasks. RANK_ADAPTIVE is the method's order.
 * SLICED is the data-slicing baseline (every rank works on slice s at step
 * s; gist.science "Technical Summary" section 1), kept for ablations only. */
typedef enum { FO_SCHED_RANK_ADAPTIVE = 0, FO_SCHED_SLICED = 1 } fo_sched;

/* How rank r gets another rank's X shard in fo_ag_gemm.
 * PEER_READ: the GEMM reads the shard straight from its owner's buffer.
 * COPY: the shard is forwarded along the ring into r's gather buffer G_r by
 *       128-bit copies, and the GEMM waits for a per-block ready flag. */
typedef enum { FO_AG_PEER_READ = 0, FO_AG_COPY = 1 } fo_ag_transport;

/* Reduce-scatter algorithm of GEMM_RS and DP_GRAD_RS (both are readings of
 * the decomposition into directed P2P chunk transfers, euno.news
 * "Methodology" item 1; the pages name a ring only for the all-gather).
 * DIRECT: each non-own partial goes straight to its owner, which adds it
 *         into its shard on arrival.
 * RING:   the running sum of chunk c travels along the ring: at step s rank
 *         r adds its partial of chunk (r - 1 - s) mod R to the sum it
 *         received from r-1 at step s-1 and forwards the result to r+1; the
 *         owner, last in the chain, adds its own partial and keeps the sum.
 *         Every forward lands in the receiver's fp32 buffer in the workspace.
 *         The additions run in step order, so the result is bitwise
 *         reproducible. Needs the rank-adaptive schedule and an interleave
 *         that runs each chunk's hops in step order: AUTO (= LOCKSTEP),
 *         LOCKSTEP or SKEWED. Not available for GEMM_AR. */
typedef enum { FO_RS_DIRECT = 0, FO_RS_RING = 1 } fo_rs_algo;

/* Storage of each W_r: KN = [K_r x N_r] row-major (default); NK = [N_r x K_r]
 * row-major (the nn.Linear weight layout, i.e. W_r transposed). */
typedef enum { FO_W_KN = 0, FO_W_NK = 1 } fo_w_layout;

/* Test hooks. DROP_TRANSFER makes fo_plan omit one transfer (the validator
 * must reject the plan). SKIP_SIGNAL makes the kernel omit the readiness
 * signal of one tile, so that a bounded wait runs out on the device.
 * DELAY_FIRST_TASK holds every tile of the first chunk task in the kernel's
 * order until inject_delay_us microseconds after its CTA started, before
 * its operands are loaded: the partials (RS/DP) or the tiles (AG) of that
 * task arrive late, and every wait for them must hold; results must not
 * change unless the delay exceeds timeout_ns. */
typedef enum {
  FO_INJECT_NONE = 0,
  FO_INJECT_DROP_TRANSFER = 1,
  FO_INJECT_SKIP_SIGNAL = 2,
  FO_INJECT_DELAY_FIRST_TASK = 3
} fo_inject;

/* Output tile of the fused kernel. AUTO: a pair of CTAs on two SMs shares
 * one 256 x 256 tile (tcgen05 cta_group::2) for bf16 inputs; fp32 inputs use
 * SINGLE. SINGLE: one CTA per SM, 128 x 256 tiles (cta_group::1). Both give
 * the same results; SINGLE exists for small problems and for comparison. */
typedef enum { FO_TILE_AUTO = 0, FO_TILE_SINGLE = 1 } fo_tile_config;

/* How the one GPU interleaves the R virtual ranks' step sequences. Every
 * choice runs each rank's tasks in that rank's schedule order and respects
 * the dependency graph; only the order across ranks differs.
 * LOCKSTEP: all ranks' step s, then step s+1 (the ranks advance together, as
 *           R GPUs would).
 * SKEWED:   rank r runs r steps behind rank 0 (slot t = s - r). Under the
 *           rank-adaptive RS order every partial of one slot is bound for the
 *           same owner, so that owner's shard stays in L2 while its partials
 *           are added.
 * RANK_MAJOR: all of rank 0's steps, then rank 1's, ...: one rank's
 *           weights (AG) or upstream gradient (DP) stay in L2 across its
 *           steps.
 * SKEWED_PAIRS: SKEWED taken two slots at a time, each rank running its
 *           two steps of the pair back to back: its weights are read once
 *           per pair, while the two owners' shards stay in L2.
 * AUTO:     SKEWED_PAIRS for GEMM_RS / GEMM_AR, RANK_MAJOR for AG_GEMM
 *           (peer read), DP_GRAD_RS and GEMM_A2A (the fastest choices on
 *           GB300 for each op; an all-to-all rank reads one X_r and one W_r
 *           for all of its steps); LOCKSTEP under the ring reduce-scatter and the copy
 *           transport, whose ring hops then run a whole step apart. */
/* Balancing of the launch's last waves. The persistent kernel deals whole
 * tiles to its units (CTA pairs or CTAs) round-robin; when the tile count is
 * not a multiple of the units, the last wave leaves most of them idle.
 * ON:   when that idle share would exceed 2% of the launch, the last
 *       partial wave plus up to two whole waves of tiles are instead cut
 *       along the reduction into equal ranges of k-blocks, one per unit; a
 *       tile cut in two is completed by the unit holding its last k-block,
 *       which adds the other part's fp32 partial (kept in the workspace).
 *       Results agree with OFF up to fp32 re-association of that tile's
 *       reduction (bit-exact in the integer mode).
 * AUTO: ON for AG_GEMM and GEMM_A2A plans whose tiles take at least 32 k-blocks and
 *       whose launch spans two or more whole waves; OFF otherwise. (Cutting
 *       costs each unit one extra store and reload of a tile; reduce-scatter
 *       tiles cut this way also wait on one another's partials, which on
 *       GB300 cost more than the balance gains.)
 * OFF:  whole tiles only. */
typedef enum { FO_TAIL_SPLIT_AUTO = 0, FO_TAIL_SPLIT_OFF = 1, FO_TAIL_SPLIT_ON = 2 } fo_tail_split;

typedef enum {
  FO_INTERLEAVE_AUTO = 0,
  FO_INTERLEAVE_LOCKSTEP = 1,
  FO_INTERLEAVE_SKEWED = 2,
  FO_INTERLEAVE_RANK_MAJOR = 3,
  FO_INTERLEAVE_SKEWED_PAIRS = 4
} fo_interleave;

/* Global GEMM sizes (M, N, K); the per-rank operands are, for each op:
 *   FO_OP_GEMM_RS    X_r [M x K/R], W_r [K/R x N] (or [N x K/R]), Y_r [M/R x N]
 *                    fp32, or bf16 with out_dtype FO_BF16
 *   FO_OP_AG_GEMM    X_r [M/R x K], W_r [K x N/R] (or [N/R x K]), Y_r [M x N/R] bf16,
 *                    optional G_r [M x K] bf16 (the gathered X)
 *   FO_OP_DP_GRAD_RS X_r [K x M], dY_r [K x N] (K = tokens), dW_r [M/R x N]
 *                    fp32, or bf16 with out_dtype FO_BF16
 *   FO_OP_GEMM_AR    X_r [M x K/R], W_r [K/R x N] (or [N x K/R]), Y_r [M x N] fp32
 *   FO_OP_GEMM_A2A   X_r [M/R x K], W_r [K x N] (or [N x K]), Y_c [M x N/R] bf16:
 *                    rows r*M/R .. (r+1)*M/R-1 of Y_c are X_r . W_r's columns
 *                    c*N/R .. (c+1)*N/R-1 (column block c = head group c)
 * With out_dtype FO_BF16 the fp32 sums are kept in the workspace and each
 * tile is rounded once (nearest even) into Y when its R-th partial lands.
 * Row block d of an RS output (rows d*M/R .. (d+1)*M/R-1 of the sum over
 * ranks) belongs to rank d. The all-gather concatenates shards in rank order.
 * GEMM_A2A uses the RS step table (the block that stays is computed last). */
typedef struct {
  int32_t op;                 /* fo_op */
  int32_t R;                  /* virtual ranks, 1..16 */
  int64_t M, N, K;
  int32_t in_dtype;           /* FO_BF16; FO_F32 (tf32 MMA) for GEMM_RS and GEMM_AR */
  int32_t out_dtype;          /* GEMM_RS / DP_GRAD_RS: FO_F32 or FO_BF16; AG_GEMM and
                                 GEMM_A2A: FO_BF16; GEMM_AR: FO_F32 */
  int32_t sched;              /* fo_sched */
  int32_t ag_transport;       /* fo_ag_transport (AG_GEMM only) */
  int32_t w_layout;           /* fo_w_layout (GEMM_RS, GEMM_AR, AG_GEMM and GEMM_A2A) */
  int32_t deterministic;      /* RS: 1 = partials are added in step order (bitwise
                                 reproducible); 0 = each add may start once the
                                 shard's first partial is stored */
  uint64_t timeout_ns;        /* bound of every device-side wait; 0 = 1 s */
  int32_t fault_inject;       /* fo_inject (tests only) */
  int32_t tile_config;        /* fo_tile_config */
  int32_t interleave;         /* fo_interleave */
  int32_t rs_algo;            /* fo_rs_algo (GEMM_RS and DP_GRAD_RS; else DIRECT) */
  int32_t trace;              /* 1: every launch records per-CTA timestamps in the
                                 workspace (fo_trace_query); 0: off */
  int32_t inject_delay_us;    /* FO_INJECT_DELAY_FIRST_TASK: 0..10^6 microseconds */
  int32_t tail_split;         /* fo_tail_split */
  int32_t reserved[1];        /* must be zero */
} fo_plan_desc;

typedef struct fo_plan_s* fo_plan_t;

/* Build and validate the schedule: per-rank step table, transfer list and
 * dependency graph (the decomposition and the rank-adaptive order cited in
 * the file header). Host only; touches no GPU. On success *out owns a new
 * plan. Returns FO_ERR_PLAN_INVARIANT when the schedule fails a check:
 * every rank's order is a permutation; RS computes its own chunk last and
 * sends nothing at its last step; AG consumes its own shard first and
 * forwards nothing at its last step; at every step the map rank -> chunk is
 * one-to-one; R(R-1) transfers; the dependency graph is acyclic and every
 * transfer precedes its consumer. (SLICED, an ablation, is checked only for
 * permutations, transfer count and acyclicity.) */
fo_status fo_plan(const fo_plan_desc* desc, fo_plan_t* out);
void fo_plan_destroy(fo_plan_t plan);

/* Copy out the R x R step table: table[r*R + s] = chunk handled by rank r at
 * step s (RS/DP: the chunk = owner of the partial; AG: the source shard). */
fo_status fo_plan_table(fo_plan_t plan, int32_t* table);

/* Copy out the transfers, 4 int32 each: (src_rank, dst_rank, chunk, step).
 * `cap` is the capacity of `out` in transfers; *n gets the count. */
fo_status fo_plan_transfers(fo_plan_t plan, int32_t* out, int32_t cap, int32_t* n);

/* Copy out the dependency edges, 4 int32 each: (rank_a, step_a, rank_b,
 * step_b) meaning task (rank_a, step_a) must finish before (rank_b, step_b)
 * may complete. `cap` in edges; *n gets the count. */
fo_status fo_plan_edges(fo_plan_t plan, int32_t* out, int32_t cap, int32_t* n);

/* Tiles the last launch with this plan cut along the reduction (the tail
 * split; 0 = none, or no launch yet). -1 for a null plan. */
int32_t fo_plan_last_split_tiles(fo_plan_t plan);

/* Copy out the order in which the kernel runs the R*R chunk tasks:
 * order[2*i] = rank, order[2*i+1] = step of the i-th task. */
fo_status fo_plan_task_order(fo_plan_t plan, int32_t* order);

/* Bytes of device workspace the launching calls need (readiness counters,
 * flags and the device status word; fp32 shard sums for a bf16 output;
 * for fp32 inputs with W as [K x N], every rank's transposed W_r;
 * under FO_RS_RING every rank's fp32 receive buffer, R x M x N x 4 bytes;
 * with trace = 1, FO_TRACE_MAX_CTAS x FO_TRACE_STAMPS timestamps; when the
 * tail split applies, one fp32 tile per split tile, sized for the 152 SMs
 * of a GB300). Never zero. */
fo_status fo_workspace_size(fo_plan_t plan, size_t* bytes);

/* Zero the workspace on `stream`. Required once before the first call that
 * uses it; calls leave it ready for the next call. */
fo_status fo_workspace_init(fo_plan_t plan, void* ws, fo_stream_t stream);

/* Flash-AG: Y_r = AllGather(X_0..X_{R-1}) . W_r for every rank r, bf16 out,
 * fp32 accumulation, rounded once (gist.science "Technical Summary" section 2,
 * Flash-All-Gather). Rank r's step s computes the rows of shard
 * (r - s) mod R. G may be NULL (no gathered copy; PEER_READ only) or an array
 * of R pointers to [M x K] bf16 buffers that receive the gathered X. Under
 * COPY, G_r is the ring-forwarded buffer the GEMM reads from. Under
 * PEER_READ it is a side output: copied by mover warps next to the GEMM, or,
 * for outputs of at most 1024 columns per rank, written from the X tiles the
 * GEMM already loads. */
fo_status fo_ag_gemm(fo_plan_t plan, const void* const* X, const void* const* W,
                     void* const* Y, void* const* G, void* ws, fo_stream_t stream);

/* Flash-RS: Y_d = sum_r (X_r . W_r)[rows of d], fp32 or bf16 (gist.science
 * "Technical Summary" section 2, Flash-Reduce-Scatter). Rank r's step s
 * computes the partial of chunk (r - 1 - s) mod R and adds it into that
 * owner's Y (FO_RS_DIRECT), or adds it to the running sum received from r-1
 * and forwards that to r+1 (FO_RS_RING); the own chunk comes last. Y is
 * overwritten. fp32 inputs run on the tf32 MMA, which reads its operands
 * K-major only: with W_r given as [K/R x N] (FO_W_KN) the call first
 * transposes every W_r into the workspace (a second launch on `stream`,
 * before the fused kernel); with [N x K/R] (FO_W_NK) it reads W_r as is. */
fo_status fo_gemm_rs(fo_plan_t plan, const void* const* X, const void* const* W,
                     void* const* Y, void* ws, fo_stream_t stream);

/* All-reduce of the partial products, as reduce-scatter then all-gather
 * (the tensor-parallel all-reduce; gist.science "Technical Summary" section 1
 * lists it beside RS and AG): Y_q = sum_r X_r . W_r for every rank q, fp32
 * [M x N]. The RS half is fo_gemm_rs into rank c's own rows of Y_c; as soon
 * as a shard tile has all R partials, the warp that added the last one
 * copies it into the same rows of every other rank's Y (the AG half), while
 * the remaining partial GEMMs still run. */
fo_status fo_gemm_ar(fo_plan_t plan, const void* const* X, const void* const* W,
                     void* const* Y, void* ws, fo_stream_t stream);

/* Flash All-to-All: the projection of Ulysses (sequence) parallelism fused
 * with its all-to-all (gist.science "Technical Summary" section 1: Ulysses
 * parallelism needs an all-to-all; section 2, "Architectural Versatility":
 * Flash All-to-All extends the method to it). Rank r holds its M/R tokens
 * X_r [M/R x K] and the whole projection W_r [K x N] ([N x K] for
 * FO_W_NK); column block c (N/R columns, head group c) of X_r . W_r belongs
 * to rank c, which stacks the blocks of all ranks in rank order:
 * Y_c [M x N/R] bf16, rows r*M/R .. (r+1)*M/R-1 from rank r (fp32
 * accumulation, rounded once). Rank r's step s computes block
 * (r - 1 - s) mod R and writes it straight into rank c's Y_c (the P2P
 * transfer); the block that stays on the rank is computed last, as in
 * Flash-RS, so no transfer trails the last compute. The blocks are
 * disjoint, so no tile waits for another. Y is overwritten. The workspace
 * holds only the status word (and the tail split's buffers). */
fo_status fo_gemm_a2a(fo_plan_t plan, const void* const* X, const void* const* W,
                      void* const* Y, void* ws, fo_stream_t stream);

/* Query-split attention with the row-parallel output projection
 * (gist.science "Technical Summary" section 2, "Architectural
 * Versatility": the attention's scores, softmax and weighted sum are
 * decomposed to put more compute beside the communication; section 1: the
 * tensor-parallel projection needs a reduce-scatter).
 * `plan`: a GEMM_RS plan with M = T tokens, N = H (the projection's output
 * width) and K = R * heads * 128, bf16 inputs, fp32 or bf16 output.
 * Rank r holds Q_r, K_r, V_r [T x heads*128] bf16 (its heads, every token;
 * head h in columns h*128 .. h*128+127) and Wo_r [heads*128 x H] ([H x
 * heads*128] with FO_W_NK); it receives O_r [T x heads*128] bf16, its
 * attention output (overwritten; kept for a backward pass), and Y_r
 * [T/R x H], rows r*T/R .. of sum_r O_r . Wo_r (overwritten).
 * Per head, O = softmax(Q K^T / sqrt(128) + mask) V over the keys; with
 * causal = 1 key j is masked for query i when j > i, with 0 nothing is.
 * The queries split into R blocks of T/R rows; rank r's step s takes block
 * (r - 1 - s) mod R, so the block that stays on the rank comes last.
 * Two launches on `stream`: fo_attention, then fo_gemm_rs of O_r . Wo_r.
 * The softmax weights are rounded to bf16 for the tensor cores' weighted
 * sum, and O once to bf16. Requires heads >= 1 and T/R a multiple of 128;
 * FO_ERR_SHAPE when K != R * heads * 128 or T/R is not; FO_ERR_INVALID_ARG
 * for another op, fp32 inputs, heads < 1 or causal not 0 or 1. Every
 * device-side wait of the attention launch gives up after 2 s (the plan's
 * timeout_ns bounds the projection's waits) and reports through
 * fo_status_query like fo_gemm_rs; a plan with FO_INJECT_SKIP_SIGNAL (tests)
 * makes one softmax signal of the attention launch go missing, so that a
 * wait runs out and the call reports FO_ERR_TIMEOUT. */
/* fo_gemm_partials for a DP_GRAD_RS plan whose A operand is the all-gather
 * of R row shards, read where they are: A_shards[s] is shard s [K/R x M]
 * bf16 (rows s*K/R .. of the gathered A [K x M], K the plan's reduction,
 * i.e. tokens), and every rank r computes P_r = A^T . B_r, B_r [K x N]
 * bf16, into P_r [R x M/R x N] fp32 like fo_gemm_partials. This is the
 * weight gradient that follows an all-gather GEMM (dW_r = AllGather(X)^T .
 * dY_r) without a gathered copy of X: the gather buffers of fo_ag_gemm can
 * be left out. Shards that lie back to back in rank order (A_shards[s] =
 * A_shards[0] + s*K/R*M elements) are read as one [K x M] tensor; others
 * through one tensor map per shard, which ran about 4% slower on GB300.
 * Requires K/R to be a multiple of 64; FO_ERR_SHAPE otherwise,
 * FO_ERR_INVALID_ARG for another op or fp32 inputs. One launch. */
fo_status fo_gemm_partials_sharded(fo_plan_t plan, const void* const* A_shards, const void* const* B,
                                   void* const* P, void* ws, fo_stream_t stream);

fo_status fo_attn_rs(fo_plan_t plan, const void* const* Q, const void* const* K, const void* const* V,
                     const void* const* Wo, void* const* O, void* const* Y, int32_t heads, int32_t causal,
                     void* ws, fo_stream_t stream);

/* The attention half of fo_attn_rs alone, one launch: O_r for every rank,
 * same arguments, layouts, checks and rounding (Wo and Y are not taken).
 * The work items, one (rank, step, head, 128-query tile) each, follow the
 * plan's task order, within a task the costlier (later) query tiles first;
 * the kernel's CTAs take them one at a time from a counter in the
 * workspace header, which the last CTA of the launch sets back to zero
 * (fo_workspace_init zeroes it; fo_status_query does after a failure). */
fo_status fo_attention(fo_plan_t plan, const void* const* Q, const void* const* K, const void* const* V,
                       void* const* O, int32_t heads, int32_t causal, void* ws, fo_stream_t stream);

/* Data-parallel weight gradient fused with its reduce-scatter:
 * dW_d = sum_r (X_r^T . dY_r)[rows of d], fp32 (gist.science "Technical
 * Summary" section 1: data parallelism needs a reduce-scatter). Same
 * schedule and reduce-scatter algorithms as fo_gemm_rs. dW is overwritten. */
fo_status fo_dp_grad_rs(fo_plan_t plan, const void* const* X, const void* const* dY,
                        void* const* dW, void* ws, fo_stream_t stream);

/* Synchronise `stream`, read the device status word from `ws` and return it
 * (FO_OK or FO_ERR_TIMEOUT). info (may be NULL) receives
 * {code, rank, step, chunk} of the first failure. A failure also re-zeroes
 * the workspace, so the plan is usable again; the outputs of the failed call
 * are undefined. */
fo_status fo_status_query(fo_plan_t plan, void* ws, fo_stream_t stream, int32_t info[4]);

/* fo_gemm_rs without a workspace, for callers that cannot allocate device
 * memory. The paper has no counterpart: this is a deployment variant of
 * fo_gemm_rs, computing the same result with the same kernel.
 *
 * Who needs it: code that runs where cudaMalloc is off limits, such as
 * inside a host callback or an allocator hook, in a process whose memory is
 * capped or pooled by another runtime, or in a plugin handed pointers but no
 * allocator. Such a caller cannot provide the workspace fo_gemm_rs takes.
 *
 * Scratch: the readiness counters and the status word live in one
 * file-scope __device__ array of FO_NOALLOC_SCRATCH_BYTES (64 KiB). Every
 * GPU that loads the library holds it until the process exits. A plan whose
 * workspace (fo_workspace_size) is larger is rejected with
 * FO_ERR_SCRATCH_LIMIT before anything is launched; 64 KiB covers, e.g.,
 * R = 8 with 8192 x 4096 outputs (16.6 KB).
 *
 * Behaviour:
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *     The caller passes inputs and outputs exactly as for fo_gemm_rs.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on the device. The address is kept for the
 *     life of the process: cudaDeviceReset (or anything else that destroys
 *     the device's primary context) invalidates it, so do not call this
 *     entry point on a device after resetting it.
 *   - Every call queries its 3R pointers (cudaPointerGetAttributes) and
 *     encodes 3R tensor maps on the host; nothing is cached in the plan.
 *   - Plan checks come first: a plan this entry point cannot run is refused
 *     before any pointer is queried or anything is enqueued.
 *   - Each call first zeroes the part of the array it uses (cudaMemsetAsync
 *     on `stream`), then launches the fused kernel.
 *   - All calls share the one array: calls that can overlap on the GPU
 *     (other streams, other host threads) race and must be serialised by the
 *     caller, e.g. by issuing them on one stream.
 *   - A device-side wait that runs out is recorded in the array and cleared
 *     by the next call; it is not reported. Use fo_gemm_rs with a workspace
 *     and fo_status_query where that report is needed.
 *   - Plans with a bf16 output return FO_ERR_DTYPE (or FO_ERR_SCRATCH_LIMIT
 *     when their shard sums exceed the array); plans with the ring
 *     reduce-scatter (FO_RS_RING), and plans with fp32 inputs and W as
 *     [K x N] (whose transposed W would need the array), return
 *     FO_ERR_UNSUPPORTED (or FO_ERR_SCRATCH_LIMIT); plans with
 *     trace = 1 return FO_ERR_SCRATCH_LIMIT (their timestamps alone fill
 *     the array). */
#define FO_NOALLOC_SCRATCH_BYTES (64 * 1024)
fo_status fo_gemm_rs_noalloc(fo_plan_t plan, const void* const* X, const void* const* W,
                             void* const* Y, fo_stream_t stream);

/* ---- tracing ------------------------------------------------------------ */

/* Timestamps (%globaltimer, ns) of the last fused-kernel launch that used
 * `ws`, for plans built with trace = 1. Per CTA, FO_TRACE_STAMPS values:
 *   [0] the CTA starts;
 *   [1] every MMA it issued has completed (leader CTAs; 0 on a pair's peer);
 *   [2..5] epilogue warp 0..3 has seen all of its stores and adds performed
 *          and released its last partial;
 *   [6] the CTA leaves;
 *   [7] 0.
 * The exposed tail of a launch, the time its transfers run past its math,
 * is max over CTAs of [2..5] minus max over CTAs of [1].
 * Copies min(cap, launched CTAs) CTAs' stamps into `stamps` (host memory,
 * cap * FO_TRACE_STAMPS values) and the launch's CTA count into *n_ctas
 * (at most FO_TRACE_MAX_CTAS CTAs are recorded). Synchronises `stream`.
 * FO_ERR_INVALID_ARG for a plan built without trace or before any launch. */
#define FO_TRACE_STAMPS 8
#define FO_TRACE_MAX_CTAS 1024
fo_status fo_trace_query(fo_plan_t plan, const void* ws, fo_stream_t stream, uint64_t* stamps, int32_t cap,
                         int32_t* n_ctas);

/* ---- measurement controls (not part of the method) --------------------- */

/* Pure-GEMM control for GEMM_RS / DP_GRAD_RS plans: the same chunk GEMM
 * tasks in the same order, but every partial is stored into its own rank's
 * [M x N] fp32 buffer P_r (no transfer, no accumulate). It doubles as the
 * per-rank GEMM where no collective follows: in a TP-SP layer each rank's
 * weight gradient (gathered activations^T . its upstream gradient) stays on
 * that rank, and a DP_GRAD_RS plan run through this call computes all R of
 * them in one launch. */
fo_status fo_gemm_partials(fo_plan_t plan, const void* const* A, const void* const* B,
                           void* const* P, void* ws, fo_stream_t stream);

/* Unfused baseline's separate reduce kernel: Y_d = sum_r P_r[rows of d] for
 * R buffers P_r [M x N] fp32 (summed in ascending r). */
fo_status fo_reduce_scatter_f32(fo_plan_t plan, const void* const* P, void* const* Y,
                                fo_stream_t stream);

/* Unfused all-gather baseline: G_r = concat(X_0..X_{R-1}) for every r, by
 * 128-bit copies (X_r [M/R x K] bf16, G_r [M x K]). */
fo_status fo_all_gather_copy(fo_plan_t plan, const void* const* X, void* const* G,
                             fo_stream_t stream);

/* Unfused all-to-all baseline for GEMM_A2A plans: Y_c[rows of r] =
 * P_r[:, column block c] for every (r, c), by 128-bit copies (P_r [M/R x N]
 * bf16, the whole projection of rank r; Y_c [M x N/R] bf16). */
fo_status fo_all_to_all_copy(fo_plan_t plan, const void* const* P, void* const* Y,
                             fo_stream_t stream);

/* Checks that each of n pointers addresses memory the current device can
 * use at that address: its own device memory, managed memory, or host memory
 * pinned or registered with CUDA. FO_OK, or FO_ERR_INVALID_ARG for pageable
 * host memory, another GPU's memory, a null array or n < 0. Pointers the
 * driver cannot classify pass. The launching calls run the same check
 * whenever their pointers change (not while `stream` captures a graph), so
 * a wrong pointer fails on the host instead of faulting in a kernel. Host
 * only; enqueues nothing. */
fo_status fo_check_device_pointers(int32_t n, const void* const* ptrs, fo_stream_t stream);

/* Number of our kernels the last launching call on this plan enqueued. */
int32_t fo_plan_last_launches(fo_plan_t plan);

const char* fo_status_string(fo_status s);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t fo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASHOVERLAP_H */
