"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer-valued inputs must match bit for bit (every fp32 partial sum is an
exact integer); random bf16 inputs must be within relative Frobenius error
1e-3 and max elementwise relative error 2e-2 (elementwise denominators
clamped at 1e-3 * rms) of the fp64 oracle. bf16 outputs (AG-GEMM) are
compared with the oracle's value rounded once to bf16.
Shapes span several tiles and ragged tails (rows per chunk, K and N that are
not multiples of the 128 x 256 x 64 tile); guard bands around every output
buffer must come back untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import WORKLOADS, ag_gemm_inputs, dp_grad_inputs, gemm_rs_inputs

pytestmark = pytest.mark.gpu

FRO_TOL = 1e-3
MAX_TOL = 2e-2
GUARD = 64          # fp32 / bf16 elements of canary on each side of an output
CANARY_F32 = -7.0e33


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _np(t):
    return t.detach().to("cpu").double().numpy()


class Guarded:
    """R output buffers, each inside a larger allocation whose head and tail
    hold a canary value."""

    def __init__(self, R, shape, dtype, dev):
        n = int(np.prod(shape))
        self.shape = shape
        self.bufs = []
        self.views = []
        for _ in range(R):
            b = torch.full((n + 2 * GUARD,), CANARY_F32, dtype=dtype, device=dev)
            self.bufs.append(b)
            self.views.append(b[GUARD:GUARD + n].view(*shape))
        self.canary = self.bufs[0][:GUARD].clone()

    def check(self):
        for b in self.bufs:
            assert torch.equal(b[:GUARD], self.canary), "write before the output buffer"
            assert torch.equal(b[-GUARD:], self.canary), "write past the output buffer"


def _ws(plan, dev):
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)
    return ws


def _status_ok(plan, ws):
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, f"device status {code} {info}"


def run_gemm_rs(dev, R, M, K, N, *, dtype="bf16", mode="int", w_layout="kn", seed=0, sched="rank_adaptive",
                deterministic=False, repeat=1, tile="auto", interleave="auto"):
    inp = gemm_rs_inputs(R, M, K, N, dtype=dtype, mode=mode, seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, in_dtype=dtype, w_layout=w_layout, sched=sched,
                     deterministic=deterministic, tile_config=tile, interleave=interleave)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if w_layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (M // R, N), torch.float32, dev)
    ws = _ws(plan, dev)
    outs = []
    for _ in range(repeat):
        B.fo_gemm_rs(plan, X, W, Y.views, ws)
        _status_ok(plan, ws)
        outs.append([_np(y) for y in Y.views])
    Y.check()
    # fp32 W as [K x N] is transposed into the workspace first: two launches
    assert B.fo_plan_last_launches(plan) == (2 if dtype == "f32" and w_layout == "kn" else 1)
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    return outs, ref


def _assert_close(got, ref):
    fro, mx, _ = oracle.rel_errors(got, ref)
    assert fro <= FRO_TOL and mx <= MAX_TOL, f"rel fro {fro:.3e}, max rel {mx:.3e}"


# ------------------------------------------------------------------ GEMM-RS

TILES = ["auto", "single"]   # CTA-pair 256x256 tiles (bf16 default) and single-CTA 128x256 tiles


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("R,M,K,N,layout", [
    (2, 256, 512, 512, "kn"),       # the 256x512x512 R=2 shape in bf16
    (4, 800, 200, 328, "kn"),       # ragged: 200 rows per chunk, K 200, N 328
    (3, 384, 64, 256, "nk"),
    (1, 128, 128, 256, "kn"),       # R = 1: plain GEMM
    (8, 1024, 136, 264, "nk"),
    (5, 640, 256, 1024, "kn"),      # several N tiles, 5 ranks
    (2, 1200, 320, 776, "nk"),      # 600-row chunks: a pair tile's second half partly out of the chunk
])
def test_gemm_rs_integer_bit_exact(dev, R, M, K, N, layout, tile):
    outs, ref = run_gemm_rs(dev, R, M, K, N, w_layout=layout, tile=tile)
    for d in range(R):
        assert np.array_equal(outs[0][d], ref[d]), f"shard {d}"


@pytest.mark.parametrize("layout", ["nk", "kn"])   # W as [N x K] (B K-major) or [K x N] (B MN-major)
@pytest.mark.parametrize("R,M,K,N", [(2, 256, 512, 512), (3, 600, 100, 132), (4, 1024, 96, 800)])
def test_gemm_rs_fp32_inputs_tf32_bit_exact(dev, R, M, K, N, layout):
    outs, ref = run_gemm_rs(dev, R, M, K, N, dtype="f32", w_layout=layout)
    for d in range(R):
        assert np.array_equal(outs[0][d], ref[d]), f"shard {d}"


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("R,M,K,N,layout", [(4, 1024, 512, 512, "kn"), (8, 1024, 200, 328, "nk")])
def test_gemm_rs_random_bf16_within_tolerance(dev, R, M, K, N, layout, tile):
    outs, ref = run_gemm_rs(dev, R, M, K, N, mode="randn", w_layout=layout, seed=2, tile=tile)
    for d in range(R):
        _assert_close(outs[0][d], ref[d])


def test_gemm_rs_deterministic_mode_is_bitwise_repeatable(dev):
    outs, ref = run_gemm_rs(dev, 4, 1024, 384, 512, mode="randn", deterministic=True, repeat=3, seed=5)
    for rep in outs[1:]:
        for d in range(4):
            assert np.array_equal(rep[d], outs[0][d])
    for d in range(4):
        _assert_close(outs[0][d], ref[d])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("interleave", ["lockstep", "skewed", "rank_major", "skewed_pairs"])
@pytest.mark.parametrize("det", [False, True])
def test_gemm_rs_every_interleave_bit_exact(dev, tile, interleave, det):
    outs, ref = run_gemm_rs(dev, 8, 2048, 136, 776, tile=tile, interleave=interleave, deterministic=det, repeat=2)
    for rep in outs:
        for d in range(8):
            assert np.array_equal(rep[d], ref[d])


def test_gemm_rs_repeated_calls_reuse_workspace(dev):
    # Counters reset themselves: many calls in a row on one workspace stay exact.
    outs, ref = run_gemm_rs(dev, 4, 512, 128, 256, repeat=5)
    for rep in outs:
        for d in range(4):
            assert np.array_equal(rep[d], ref[d])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("det", [False, True])
def test_gemm_rs_one_cta_holds_first_and_second_partial_of_a_tile(dev, det, tile):
    # One m-tile per chunk and exactly one n-tile per SM (per SM pair): the
    # CTA that stores a shard tile's first partial is the one that adds its
    # second partial next, so the epilogue must publish its own deferred
    # partial before it waits for it.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    units = sms if tile == "single" else sms // 2
    R, M, K, N = 2, 2 * (128 if tile == "single" else 256), 64, 256 * units
    outs, ref = run_gemm_rs(dev, R, M, K, N, deterministic=det, tile=tile)
    for d in range(R):
        assert np.array_equal(outs[0][d], ref[d])


def test_gemm_rs_sliced_ablation_same_result(dev):
    outs, ref = run_gemm_rs(dev, 4, 512, 128, 512, sched="sliced")
    for d in range(4):
        assert np.array_equal(outs[0][d], ref[d])


def test_gemm_rs_new_buffers_after_cached_call(dev):
    R, M, K, N = 2, 256, 128, 256
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    ws = _ws(plan, dev)
    for seed in (1, 2):
        inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=seed)
        X = [x.to(dev) for x in inp["X"]]
        W = [w.to(dev) for w in inp["W"]]
        Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
        B.fo_gemm_rs(plan, X, W, Y, ws)
        _status_ok(plan, ws)
        ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for d in range(R):
            assert np.array_equal(_np(Y[d]), ref[d])


# ------------------------------------------------------------------ all-reduce and bf16 output

@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("interleave", ["lockstep", "skewed", "skewed_pairs"])
@pytest.mark.parametrize("R,M,K,N", [(4, 1024, 136, 520), (2, 600, 200, 264), (8, 2048, 64, 256), (1, 256, 128, 256)])
def test_gemm_ar_integer_bit_exact(dev, tile, interleave, R, M, K, N):
    # RS into each owner's rows of its full output, then every finished
    # shard tile copied to all other ranks: every rank holds the whole sum.
    plan = B.fo_plan("gemm_ar", R, M, N, K * R, tile_config=tile, interleave=interleave)
    ws = _ws(plan, dev)
    Y = Guarded(R, (M, N), torch.float32, dev)
    for seed in (7, 8):
        inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=seed)
        X = [x.to(dev) for x in inp["X"]]
        W = [w.to(dev) for w in inp["W"]]
        B.fo_gemm_ar(plan, X, W, Y.views, ws)
        _status_ok(plan, ws)
        ref = oracle.gemm_ar([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for q in range(R):
            assert np.array_equal(_np(Y.views[q]), ref[q]), f"rank {q}"
    Y.check()


def test_gemm_ar_random_bf16_within_tolerance(dev):
    R, M, K, N = 4, 1024, 512, 512
    inp = gemm_rs_inputs(R, M, K, N, mode="randn", seed=3)
    plan = B.fo_plan("gemm_ar", R, M, N, K * R)
    ws = _ws(plan, dev)
    Y = [torch.empty(M, N, device=dev) for _ in range(R)]
    B.fo_gemm_ar(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y, ws)
    _status_ok(plan, ws)
    ref = oracle.gemm_ar([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for q in range(R):
        _assert_close(_np(Y[q]), ref[q])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("mode", ["int", "randn"])
def test_gemm_rs_bf16_output_is_rounded_once(dev, tile, mode):
    R, M, K, N = 4, 800, 200, 328
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, out_dtype="bf16", tile_config=tile)
    ws = _ws(plan, dev)
    Y = Guarded(R, (M // R, N), torch.bfloat16, dev)
    for seed in (1, 2):
        inp = gemm_rs_inputs(R, M, K, N, mode=mode, seed=seed)
        B.fo_gemm_rs(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
        _status_ok(plan, ws)
        ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for d in range(R):
            want = oracle.round_bf16(ref[d])
            if mode == "int":
                assert np.array_equal(_np(Y.views[d]), want)
            else:
                _assert_close(_np(Y.views[d]), want)
    Y.check()


def test_dp_grad_rs_bf16_output(dev):
    R, T, M, N = 4, 200, 800, 328
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=5)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, out_dtype="bf16")
    ws = _ws(plan, dev)
    dW = Guarded(R, (M // R, N), torch.bfloat16, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW.views, ws)
    _status_ok(plan, ws)
    dW.check()
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        assert np.array_equal(_np(dW.views[d]), oracle.round_bf16(ref[d]))


# ------------------------------------------------------------------ AG-GEMM

def run_ag(dev, R, M, K, N, *, mode="int", layout="kn", seed=1, tile="auto", interleave="auto"):
    inp = ag_gemm_inputs(R, M, K, N // R, mode=mode, seed=seed)
    plan = B.fo_plan("ag_gemm", R, M, N, K, w_layout=layout, tile_config=tile, interleave=interleave)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (M, N // R), torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_ag_gemm(plan, X, W, Y.views, None, ws)
    _status_ok(plan, ws)
    Y.check()
    ref, _ = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    return [_np(y) for y in Y.views], ref


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("R,M,K,N,layout", [
    (4, 512, 256, 512, "kn"),
    (2, 400, 200, 336, "kn"),       # ragged: 200-row shards, K 200, 168 columns per rank
    (3, 384, 64, 768, "nk"),
    (1, 256, 128, 256, "kn"),
    (2, 1200, 136, 1040, "nk"),     # 600-row shards, 520 columns per rank
])
def test_ag_gemm_integer_bit_exact(dev, R, M, K, N, layout, tile):
    got, ref = run_ag(dev, R, M, K, N, layout=layout, tile=tile)
    for r in range(R):
        assert np.array_equal(got[r], oracle.round_bf16(ref[r])), f"rank {r}"


def run_ag_gather(dev, R, M, K, N, *, transport, tile="auto", layout="kn", seeds=(1,), inject="none", timeout_ns=0):
    plan = B.fo_plan("ag_gemm", R, M, N, K, w_layout=layout, tile_config=tile, ag_transport=transport,
                     fault_inject=inject, timeout_ns=timeout_ns)
    ws = _ws(plan, dev)
    Y = Guarded(R, (M, N // R), torch.bfloat16, dev)
    G = Guarded(R, (M, K), torch.bfloat16, dev)
    X = [torch.empty(M // R, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    W = [torch.empty((K, N // R) if layout == "kn" else (N // R, K), dtype=torch.bfloat16, device=dev)
         for _ in range(R)]
    results = []
    for seed in seeds:
        inp = ag_gemm_inputs(R, M, K, N // R, mode="int", seed=seed)
        for r in range(R):        # same buffers, new contents: stale data from a previous call must not pass
            X[r].copy_(inp["X"][r])
            W[r].copy_(inp["W"][r] if layout == "kn" else inp["W"][r].t())
        B.fo_ag_gemm(plan, X, W, Y.views, G.views, ws)
        code, info = B.fo_status_query(plan, ws)
        results.append((code, info, [_np(y) for y in Y.views], [_np(g) for g in G.views], inp))
    Y.check()
    G.check()
    return results


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("transport", ["copy", "peer_read"])
@pytest.mark.parametrize("R,M,K,N,layout", [(4, 1024, 256, 512, "kn"), (2, 400, 200, 336, "nk"),
                                             (3, 600, 136, 768, "kn"),
                                             (2, 400, 136, 2560, "kn"), (4, 1000, 200, 5120, "nk")])
def test_ag_gemm_gather_buffers_bit_exact(dev, tile, transport, R, M, K, N, layout):
    # copy: shards travel the ring into G_r and the GEMM of steps >= 1 reads
    # them there; peer_read: G_r is a side output, written from the GEMM's
    # loaded X tiles (outputs of <= 1024 columns per rank) or by mover warps
    # (the last two shapes). Either way Y_r and G_r are exact; two calls in a
    # row with new inputs on one workspace.
    for code, info, Y, G, inp in run_ag_gather(dev, R, M, K, N, transport=transport, tile=tile, layout=layout,
                                               seeds=(1, 2)):
        assert code == 0, info
        ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for r in range(R):
            assert np.array_equal(Y[r], oracle.round_bf16(ref[r])), f"Y rank {r}"
            assert np.array_equal(G[r], gathered), f"G rank {r}"


def test_ag_copy_missing_ready_flag_times_out(dev):
    R, M, K, N = 2, 512, 128, 512
    (code, info, _, _, _), = run_ag_gather(dev, R, M, K, N, transport="copy", inject="skip_signal",
                                           timeout_ns=20_000_000)
    assert code == B.FO_ERR_TIMEOUT
    assert info == [B.FO_ERR_TIMEOUT, 1, 1, 0]      # rank 1 waits at step 1 for shard 0
    # the workspace was reset by the status query: a clean plan runs exactly
    (code, info, Y, G, inp), = run_ag_gather(dev, R, M, K, N, transport="copy")
    assert code == 0
    ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for r in range(R):
        assert np.array_equal(Y[r], oracle.round_bf16(ref[r]))


@pytest.mark.parametrize("interleave", ["skewed", "rank_major"])
def test_ag_gemm_interleaves_bit_exact(dev, interleave):
    got, ref = run_ag(dev, 4, 1024, 136, 1056, interleave=interleave)
    for r in range(4):
        assert np.array_equal(got[r], oracle.round_bf16(ref[r]))


@pytest.mark.parametrize("R,M,K,N", [(4, 1024, 512, 1024), (2, 400, 200, 336)])
def test_ag_gemm_random_bf16_within_tolerance(dev, R, M, K, N):
    got, ref = run_ag(dev, R, M, K, N, mode="randn")
    for r in range(R):
        _assert_close(got[r], oracle.round_bf16(ref[r]))


# ------------------------------------------------------------------ DP grad

def run_dp(dev, R, T, M, N, *, mode="int", seed=3, tile="auto", interleave="auto"):
    inp = dp_grad_inputs(R, T, M, N, mode=mode, seed=seed)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, tile_config=tile, interleave=interleave)
    X = [x.to(dev) for x in inp["X"]]
    dY = [y.to(dev) for y in inp["dY"]]
    dW = Guarded(R, (M // R, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, X, dY, dW.views, ws)
    _status_ok(plan, ws)
    dW.check()
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    return [_np(w) for w in dW.views], ref


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("R,T,M,N", [(1, 128, 256, 256), (2, 256, 256, 256), (4, 200, 800, 328), (8, 128, 1024, 256)])
def test_dp_grad_rs_integer_bit_exact(dev, R, T, M, N, tile):
    got, ref = run_dp(dev, R, T, M, N, tile=tile)
    for d in range(R):
        assert np.array_equal(got[d], ref[d]), f"shard {d}"


@pytest.mark.parametrize("interleave", ["lockstep", "skewed", "rank_major"])
def test_dp_grad_rs_interleaves_bit_exact(dev, interleave):
    got, ref = run_dp(dev, 4, 200, 800, 328, interleave=interleave)
    for d in range(4):
        assert np.array_equal(got[d], ref[d])


def test_dp_grad_rs_random_bf16_within_tolerance(dev):
    got, ref = run_dp(dev, 4, 512, 1024, 512, mode="randn")
    for d in range(4):
        _assert_close(got[d], ref[d])


# ------------------------------------------------------------------ controls

def test_partials_control_stores_each_ranks_gemm(dev):
    R, M, K, N = 4, 512, 192, 256
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=9)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]
    P = [torch.empty(M, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_partials(plan, X, W, P, ws)
    _status_ok(plan, ws)
    for r in range(R):
        assert np.array_equal(_np(P[r]), _np(inp["X"][r]) @ _np(inp["W"][r]))
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    B.fo_reduce_scatter_f32(plan, P, Y)
    torch.cuda.synchronize()
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        assert np.array_equal(_np(Y[d]), ref[d])



def _place_shards(shards, placement, dev):
    """The shards on the device: separate allocations, back to back in one
    buffer, or one buffer with a 64-row gap after each shard."""
    if placement == "separate":
        return [a.to(dev) for a in shards]
    if placement == "back_to_back":
        return list(torch.cat(shards).to(dev).split(shards[0].shape[0]))
    rows, gap = shards[0].shape[0], 64
    buf = torch.zeros(len(shards) * (rows + gap), shards[0].shape[1], dtype=shards[0].dtype, device=dev)
    views = [buf[s * (rows + gap):s * (rows + gap) + rows] for s in range(len(shards))]
    for v, a in zip(views, shards):
        v.copy_(a)
    return views


@pytest.mark.parametrize("placement", ["separate", "back_to_back", "spaced"])
@pytest.mark.parametrize("R,T,M,N", [(2, 128, 256, 64), (4, 768, 800, 328), (8, 1024, 512, 136)])
def test_partials_sharded_reads_the_gather_in_place(dev, R, T, M, N, placement):
    """fo_gemm_partials_sharded: A = AllGather of R row shards of [T/R x M],
    read where the shards lie (separate allocations: one tensor map per
    shard; back to back: one map; one stride apart: one 3-D map); P_r =
    A^T . dY_r for every rank, bit for bit (integer inputs make the fp32
    sums exact)."""
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=11)
    shards = list(inp["X"][0].split(T // R))
    A = _place_shards(shards, placement, dev)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T)
    P = Guarded(R, (M, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_partials_sharded(plan, A, [y.to(dev) for y in inp["dY"]], P.views, ws)
    _status_ok(plan, ws)
    P.check()
    G = oracle.all_gather_rows([_np(a) for a in shards])
    ref = oracle.weight_grads([G] * R, [_np(y) for y in inp["dY"]])
    for r in range(R):
        assert np.array_equal(_np(P.views[r]), ref[r]), f"rank {r}"


def test_partials_sharded_random_bf16_within_tolerance(dev):
    R, T, M, N = 4, 2048, 1024, 512
    inp = dp_grad_inputs(R, T, M, N, mode="randn", seed=12)
    shards = list(inp["X"][0].split(T // R))
    plan = B.fo_plan("dp_grad_rs", R, M, N, T)
    P = [torch.empty(M, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_partials_sharded(plan, [a.to(dev) for a in shards], [y.to(dev) for y in inp["dY"]], P, ws)
    _status_ok(plan, ws)
    G = oracle.all_gather_rows([_np(a) for a in shards])
    ref = oracle.weight_grads([G] * R, [_np(y) for y in inp["dY"]])
    for r in range(R):
        _assert_close(_np(P[r]), ref[r])

def test_all_gather_copy(dev):
    R, M, K, N = 4, 512, 256, 512
    inp = ag_gemm_inputs(R, M, K, N // R, mode="randn", seed=4)
    plan = B.fo_plan("ag_gemm", R, M, N, K)
    X = [x.to(dev) for x in inp["X"]]
    G = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    B.fo_all_gather_copy(plan, X, G)
    torch.cuda.synchronize()
    want = oracle.all_gather_rows([_np(x) for x in inp["X"]])
    for r in range(R):
        assert np.array_equal(_np(G[r]), want)


# ------------------------------------------------------------------ failure detection

def test_missing_signal_times_out_and_workspace_recovers(dev):
    R, M, K, N = 2, 256, 128, 256
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=0)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    bad = B.fo_plan("gemm_rs", R, M, N, K * R, fault_inject="skip_signal", timeout_ns=20_000_000)
    ws = _ws(bad, dev)
    B.fo_gemm_rs(bad, X, W, Y, ws)
    code, info = B.fo_status_query(bad, ws)
    assert code == B.FO_ERR_TIMEOUT
    # chunk 0 gets its second partial from rank 0 at step 1 (its own chunk, last)
    assert info == [B.FO_ERR_TIMEOUT, 0, 1, 0]
    good = B.fo_plan("gemm_rs", R, M, N, K * R)
    B.fo_gemm_rs(good, X, W, Y, ws)
    _status_ok(good, ws)
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        assert np.array_equal(_np(Y[d]), ref[d])


# ------------------------------------------------------------------ full-size workloads (sampled rows)

def _sample_rows(rng, n, k=48):
    rows = rng.choice(n, size=min(k, n), replace=False)
    rows[:2] = [0, n - 1]
    return np.sort(rows)


def test_full_size_gemm_rs_down_proj(dev):
    w = WORKLOADS["gemm_rs_down_r8_t8192_k1792_n4096"]
    R, M, K, N = w.R, w.dims["M"], w.dims["K"], w.dims["N"]
    inp = w.make()
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    X = [x.to(dev) for x in inp["X"]]
    W = [x.to(dev) for x in inp["W"]]
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_rs(plan, X, W, Y, ws)
    _status_ok(plan, ws)
    Xn = [_np(x) for x in inp["X"]]
    Wn = [_np(x) for x in inp["W"]]
    rng = np.random.default_rng(0)
    for d in range(R):
        rows = _sample_rows(rng, M // R)
        _assert_close(_np(Y[d][torch.as_tensor(rows, device=dev)]), oracle.gemm_rs_rows(Xn, Wn, d, rows))


def test_full_size_ag_gemm_qkv(dev):
    w = WORKLOADS["ag_gemm_qkv_r4_s4096_h4096_n3072"]
    R, M, K, Nr = w.R, w.dims["M"], w.dims["K"], w.dims["N"]
    inp = w.make()
    plan = B.fo_plan("ag_gemm", R, M, Nr * R, K)
    X = [x.to(dev) for x in inp["X"]]
    W = [x.to(dev) for x in inp["W"]]
    Y = [torch.empty(M, Nr, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_ag_gemm(plan, X, W, Y, None, ws)
    _status_ok(plan, ws)
    Xn = [_np(x) for x in inp["X"]]
    Wn = [_np(x) for x in inp["W"]]
    rng = np.random.default_rng(1)
    for r in range(R):
        rows = _sample_rows(rng, M)
        got = _np(Y[r][torch.as_tensor(rows, device=dev)])
        _assert_close(got, oracle.round_bf16(oracle.ag_gemm_rows(Xn, Wn, r, rows)))


def test_full_size_dp_grad(dev):
    w = WORKLOADS["dp_grad_rs_r8_t4096_4096x4096"]
    R, T, M, N = w.R, w.dims["T"], w.dims["M"], w.dims["N"]
    inp = w.make()
    plan = B.fo_plan("dp_grad_rs", R, M, N, T)
    X = [x.to(dev) for x in inp["X"]]
    dY = [x.to(dev) for x in inp["dY"]]
    dW = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, X, dY, dW, ws)
    _status_ok(plan, ws)
    Xn = [_np(x) for x in inp["X"]]
    dYn = [_np(x) for x in inp["dY"]]
    rng = np.random.default_rng(3)
    for d in range(R):
        rows = _sample_rows(rng, M // R, 16)
        _assert_close(_np(dW[d][torch.as_tensor(rows, device=dev)]), oracle.dp_grad_rs_rows(Xn, dYn, d, rows))
