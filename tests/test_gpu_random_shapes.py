"""Seeded random shapes for every op (reduce-scatter with bf16 and fp32
inputs, all-gather, DP gradient, the weight gradient over token shards,
all-reduce, all-to-all): R from 1 to 16, ragged rows, K and N,
either tile configuration, any interleave, both weight layouts and output
dtypes, with the tail split forced on in about half the draws. Integer inputs, so every result must equal the oracle bit for bit
(bf16 outputs: the oracle rounded once); guard bands around every output.
Dimensions are multiples of 8 so that every row of every operand starts on
a 16-byte boundary, as the library requires.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import ag_gemm_inputs, dp_grad_inputs, gemm_rs_inputs
from test_gpu_parity import Guarded, _np, _place_shards, _status_ok, _ws

pytestmark = pytest.mark.gpu

CASES = 25
INTERLEAVES = ["auto", "lockstep", "skewed", "rank_major", "skewed_pairs"]
SPLITS = ["auto", "on"]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _draw(seed):
    g = np.random.default_rng(seed)
    R = int(g.integers(1, 17))
    rows = 8 * int(g.integers(1, 41))          # rows per rank: 8 .. 320
    K = 8 * int(g.integers(1, 49))             # 8 .. 384
    N = 8 * int(g.integers(1, 65))             # 8 .. 512
    return g, R, rows, K, N


@pytest.mark.parametrize("seed", range(CASES))
def test_random_gemm_rs(dev, seed):
    g, R, rows, Kr, N = _draw(1000 + seed)
    M = R * rows
    layout = ["kn", "nk"][int(g.integers(2))]
    out = ["f32", "bf16"][int(g.integers(2))]
    tile = ["auto", "single"][int(g.integers(2))]
    il = INTERLEAVES[int(g.integers(len(INTERLEAVES)))]
    det = bool(g.integers(2))
    split = SPLITS[int(g.integers(2))]
    inp = gemm_rs_inputs(R, M, Kr, N, mode="int", seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, Kr * R, w_layout=layout, out_dtype=out, tile_config=tile,
                     interleave=il, deterministic=det, tail_split=split)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (rows, N), torch.float32 if out == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_gemm_rs(plan, X, W, Y.views, ws)
        _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        want = ref[d] if out == "f32" else oracle.round_bf16(ref[d])
        assert np.array_equal(_np(Y.views[d]), want), f"R={R} M={M} K={Kr} N={N} {layout} {out} {tile} {il} {split} shard {d}"


@pytest.mark.parametrize("seed", range(CASES))
def test_random_ag_gemm(dev, seed):
    g, R, rows, K, Nr = _draw(2000 + seed)
    M = R * rows
    layout = ["kn", "nk"][int(g.integers(2))]
    tile = ["auto", "single"][int(g.integers(2))]
    il = INTERLEAVES[int(g.integers(len(INTERLEAVES)))]
    transport = ["peer_read", "copy"][int(g.integers(2))]
    with_g = transport == "copy" or bool(g.integers(2))
    split = SPLITS[int(g.integers(2))]
    inp = ag_gemm_inputs(R, M, K, Nr, mode="int", seed=seed)
    plan = B.fo_plan("ag_gemm", R, M, Nr * R, K, w_layout=layout, tile_config=tile, interleave=il,
                     ag_transport=transport, tail_split=split)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (M, Nr), torch.bfloat16, dev)
    G = Guarded(R, (M, K), torch.bfloat16, dev) if with_g else None
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_ag_gemm(plan, X, W, Y.views, G.views if G else None, ws)
        _status_ok(plan, ws)
    Y.check()
    ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    what = f"R={R} M={M} K={K} N_r={Nr} {layout} {tile} {il} {transport} G={with_g} {split}"
    for r in range(R):
        assert np.array_equal(_np(Y.views[r]), oracle.round_bf16(ref[r])), f"{what} rank {r}"
    if G:
        G.check()
        for r in range(R):
            assert np.array_equal(_np(G.views[r]), gathered), f"{what} gather buffer {r}"


@pytest.mark.parametrize("seed", range(CASES))
def test_random_dp_grad_rs(dev, seed):
    g, R, rows, T, N = _draw(3000 + seed)
    M = R * rows
    tile = ["auto", "single"][int(g.integers(2))]
    il = INTERLEAVES[int(g.integers(len(INTERLEAVES)))]
    out = ["f32", "bf16"][int(g.integers(2))]
    split = SPLITS[int(g.integers(2))]
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=seed)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, tile_config=tile, interleave=il, out_dtype=out, tail_split=split)
    dW = Guarded(R, (rows, N), torch.float32 if out == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW.views, ws)
    _status_ok(plan, ws)
    dW.check()
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        want = ref[d] if out == "f32" else oracle.round_bf16(ref[d])
        assert np.array_equal(_np(dW.views[d]), want), f"R={R} T={T} M={M} N={N} {tile} {il} {out} {split} shard {d}"



@pytest.mark.parametrize("seed", range(CASES))
def test_random_partials_sharded(dev, seed):
    # The gathered A given as R token shards (64-row multiples): separate
    # allocations, back to back, or one stride apart; P_r = AllGather(A)^T . dY_r.
    g, R, rows, _, N = _draw(9000 + seed)
    M = R * rows
    T = R * 64 * int(g.integers(1, 5))
    tile = ["auto", "single"][int(g.integers(2))]
    il = INTERLEAVES[int(g.integers(len(INTERLEAVES)))]
    split = SPLITS[int(g.integers(2))]
    placement = ["separate", "back_to_back", "spaced"][int(g.integers(3))]
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=seed)
    whole = inp["X"][0]
    A = _place_shards(list(whole.split(T // R)), placement, dev)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, tile_config=tile, interleave=il, tail_split=split)
    P = Guarded(R, (M, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_partials_sharded(plan, A, [y.to(dev) for y in inp["dY"]], P.views, ws)
    _status_ok(plan, ws)
    P.check()
    ref = oracle.weight_grads([oracle.all_gather_rows([_np(a) for a in whole.split(T // R)])] * R,
                              [_np(y) for y in inp["dY"]])
    for r in range(R):
        assert np.array_equal(_np(P.views[r]), ref[r]), \
            f"R={R} T={T} M={M} N={N} {tile} {il} {split} {placement} rank {r}"

@pytest.mark.parametrize("seed", range(CASES))
def test_random_gemm_ar(dev, seed):
    g, R, rows, Kr, N = _draw(4000 + seed)
    M = R * rows
    tile = ["auto", "single"][int(g.integers(2))]
    il = ["auto", "lockstep", "skewed", "skewed_pairs"][int(g.integers(4))]
    split = SPLITS[int(g.integers(2))]
    inp = gemm_rs_inputs(R, M, Kr, N, mode="int", seed=seed)
    plan = B.fo_plan("gemm_ar", R, M, N, Kr * R, tile_config=tile, interleave=il, tail_split=split)
    Y = Guarded(R, (M, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_ar(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
    _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_ar([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for q in range(R):
        assert np.array_equal(_np(Y.views[q]), ref[q]), f"R={R} M={M} K={Kr} N={N} {tile} {il} {split} rank {q}"


@pytest.mark.parametrize("seed", range(CASES))
def test_random_gemm_a2a(dev, seed):
    g, R, rows, K, Nc = _draw(8000 + seed)       # Nc: columns of one block (head group)
    M, N = R * rows, R * Nc
    layout = ["kn", "nk"][int(g.integers(2))]
    tile = ["auto", "single"][int(g.integers(2))]
    il = INTERLEAVES[int(g.integers(len(INTERLEAVES)))]
    sched = ["rank_adaptive", "sliced"][int(g.integers(2))]
    split = SPLITS[int(g.integers(2))]
    inp = ag_gemm_inputs(R, M, K, N, mode="int", seed=seed)
    plan = B.fo_plan("gemm_a2a", R, M, N, K, w_layout=layout, tile_config=tile, interleave=il, sched=sched,
                     tail_split=split)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (M, Nc), torch.bfloat16, dev)
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_gemm_a2a(plan, X, W, Y.views, ws)
        _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_a2a([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    what = f"R={R} M={M} K={K} N={N} {layout} {tile} {il} {sched} {split}"
    for c in range(R):
        assert np.array_equal(_np(Y.views[c]), oracle.round_bf16(ref[c])), f"{what} rank {c}"


@pytest.mark.parametrize("seed", range(CASES // 2))
def test_random_gemm_rs_fp32_inputs(dev, seed):
    # fp32 inputs on the tf32 MMA, W in either layout ([K x N] is transposed
    # into the workspace first); K and N multiples of 4 keep fp32 rows on
    # 16-byte boundaries.
    g, R, rows, Kr, N = _draw(9000 + seed)
    M = R * rows
    layout = ["kn", "nk"][int(g.integers(2))]
    split = SPLITS[int(g.integers(2))]
    inp = gemm_rs_inputs(R, M, Kr, N, dtype="f32", mode="int", seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, Kr * R, in_dtype="f32", w_layout=layout, tail_split=split)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    Y = Guarded(R, (rows, N), torch.float32, dev)
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_gemm_rs(plan, X, W, Y.views, ws)
        _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        assert np.array_equal(_np(Y.views[d]), ref[d]), f"R={R} M={M} K={Kr} N={N} {layout} {split} shard {d}"


# ---------------------------------------------------------------- random data
# The same draws with normal-distributed inputs, held to the stated
# tolerances: relative Frobenius error <= 1e-3 and elementwise relative error
# <= 2e-2 against the fp64 oracle (rounded once to bf16 for bf16 outputs).
RANDN_CASES = 8
FRO_TOL, MAX_TOL = 1e-3, 2e-2


def _close(got, want, what):
    fro, mx, _ = oracle.rel_errors(got, want)
    assert fro <= FRO_TOL and mx <= MAX_TOL, f"{what}: rel fro {fro:.3e}, max rel {mx:.3e}"


@pytest.mark.parametrize("seed", range(RANDN_CASES))
def test_random_gemm_rs_randn(dev, seed):
    g, R, rows, Kr, N = _draw(5000 + seed)
    M = R * rows
    out = ["f32", "bf16"][int(g.integers(2))]
    split = SPLITS[int(g.integers(2))]
    inp = gemm_rs_inputs(R, M, Kr, N, mode="randn", seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, Kr * R, out_dtype=out, tail_split=split)
    Y = Guarded(R, (rows, N), torch.float32 if out == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_rs(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
    _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        want = ref[d] if out == "f32" else oracle.round_bf16(ref[d])
        _close(_np(Y.views[d]), want, f"R={R} M={M} K={Kr} N={N} {out} {split} shard {d}")


@pytest.mark.parametrize("seed", range(RANDN_CASES))
def test_random_ag_gemm_randn(dev, seed):
    g, R, rows, K, Nr = _draw(6000 + seed)
    M = R * rows
    split = SPLITS[int(g.integers(2))]
    inp = ag_gemm_inputs(R, M, K, Nr, mode="randn", seed=seed)
    plan = B.fo_plan("ag_gemm", R, M, Nr * R, K, tail_split=split)
    Y = Guarded(R, (M, Nr), torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_ag_gemm(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, None, ws)
    _status_ok(plan, ws)
    Y.check()
    ref, _ = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for r in range(R):
        _close(_np(Y.views[r]), oracle.round_bf16(ref[r]), f"R={R} M={M} K={K} N_r={Nr} {split} rank {r}")


@pytest.mark.parametrize("seed", range(RANDN_CASES))
def test_random_dp_grad_rs_randn(dev, seed):
    g, R, rows, T, N = _draw(7000 + seed)
    M = R * rows
    out = ["f32", "bf16"][int(g.integers(2))]
    split = SPLITS[int(g.integers(2))]
    inp = dp_grad_inputs(R, T, M, N, mode="randn", seed=seed)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, out_dtype=out, tail_split=split)
    dW = Guarded(R, (rows, N), torch.float32 if out == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW.views, ws)
    _status_ok(plan, ws)
    dW.check()
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        want = ref[d] if out == "f32" else oracle.round_bf16(ref[d])
        _close(_np(dW.views[d]), want, f"R={R} T={T} M={M} N={N} {out} {split} shard {d}")


@pytest.mark.parametrize("seed", range(RANDN_CASES))
def test_random_gemm_a2a_randn(dev, seed):
    g, R, rows, K, Nc = _draw(10000 + seed)
    M, N = R * rows, R * Nc
    split = SPLITS[int(g.integers(2))]
    inp = ag_gemm_inputs(R, M, K, N, mode="randn", seed=seed)
    plan = B.fo_plan("gemm_a2a", R, M, N, K, tail_split=split)
    Y = Guarded(R, (M, Nc), torch.bfloat16, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_a2a(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
    _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_a2a([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for c in range(R):
        _close(_np(Y.views[c]), oracle.round_bf16(ref[c]), f"R={R} M={M} K={K} N={N} {split} rank {c}")
