"""GPU parity of the tail split: when a launch's tiles leave its last wave
mostly idle, the last partial wave plus two whole waves of tiles are cut along
the reduction and dealt out evenly; a tile cut in two is completed by the
unit holding its last k-block, which adds the other part's fp32 partial.

Integer-valued inputs stay bit-exact against the oracle (every fp32 sum is
exact whatever the order); random inputs stay within the tolerance. Each
shape below is chosen so that a GB300 (76 CTA pairs or 152 CTAs) does cut
tiles (with the split forced on where AUTO would not cut), which the test
checks through fo_plan_last_split_tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import ag_gemm_inputs, dp_grad_inputs, gemm_rs_inputs

pytestmark = pytest.mark.gpu

FRO_TOL = 1e-3
MAX_TOL = 2e-2
GUARD = 64
CANARY = -7.0e33


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _np(t):
    return t.detach().to("cpu").double().numpy()


def _guarded(R, shape, dtype, dev):
    n = int(np.prod(shape))
    bufs = [torch.full((n + 2 * GUARD,), CANARY, dtype=dtype, device=dev) for _ in range(R)]
    return bufs, [b[GUARD:GUARD + n].view(*shape) for b in bufs]


def _guards_intact(bufs):
    ref = bufs[0][:GUARD].clone()
    for b in bufs:
        assert torch.equal(b[:GUARD], ref) and torch.equal(b[-GUARD:], ref), "write outside an output"


def _ws(plan, dev):
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)
    return ws


def _status_ok(plan, ws):
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, f"device status {code} {info}"


def _close(got, ref):
    fro, mx, _ = oracle.rel_errors(got, ref)
    assert fro <= FRO_TOL and mx <= MAX_TOL, f"rel fro {fro:.3e}, max rel {mx:.3e}"


def run_rs(dev, R, M, K, N, *, mode="int", dtype="bf16", layout="kn", out_dtype="f32", seed=0, repeat=2, **kw):
    inp = gemm_rs_inputs(R, M, K, N, dtype=dtype, mode=mode, seed=seed)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    outs = {}
    for split in ("on", "off"):
        plan = B.fo_plan("gemm_rs", R, M, N, K * R, in_dtype=dtype, w_layout=layout, out_dtype=out_dtype,
                         tail_split=split, **kw)
        bufs, Y = _guarded(R, (M // R, N), torch.float32 if out_dtype == "f32" else torch.bfloat16, dev)
        ws = _ws(plan, dev)
        for _ in range(repeat):   # the second call reuses the split counters
            B.fo_gemm_rs(plan, X, W, Y, ws)
            _status_ok(plan, ws)
        _guards_intact(bufs)
        outs[split] = ([_np(y) for y in Y], B.fo_plan_last_split_tiles(plan))
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    return outs, ref


@pytest.mark.parametrize("R,M,K,N,tile,kw", [
    (4, 1024, 256, 1280, "auto", {}),                        # 80 pair tiles: one wave + 4, all cut
    (4, 1024, 448, 2560, "auto", {}),                        # 160 pair tiles, all cut (2 waves + 8)
    (4, 1024, 448, 3840, "auto", {}),                        # 240 pair tiles: 76 whole + 164 cut
    (4, 1000, 200, 1240, "auto", {}),                        # ragged rows, K and N
    (4, 1024, 256, 2560, "single", {}),                      # 160 single-CTA tiles on 152 CTAs
    (4, 1024, 256, 1280, "auto", dict(deterministic=True)),
    (4, 1024, 256, 1280, "auto", dict(rs_algo="ring")),
    (4, 1024, 256, 1280, "auto", dict(interleave="lockstep")),
])
def test_split_gemm_rs_integer_bit_exact(dev, R, M, K, N, tile, kw):
    outs, ref = run_rs(dev, R, M, K, N, tile_config=tile, **kw)
    (got, split), (off, nosplit) = outs["on"], outs["off"]
    assert split > 0 and nosplit == 0
    for d in range(R):
        assert np.array_equal(got[d], ref[d]), f"shard {d}"
        assert np.array_equal(off[d], ref[d])


@pytest.mark.parametrize("layout", ["nk", "kn"])
def test_split_gemm_rs_tf32_bit_exact(dev, layout):
    outs, ref = run_rs(dev, 2, 512, 256, 5120, dtype="f32", layout=layout)   # 160 single-CTA tiles
    assert outs["on"][1] > 0
    for d in range(2):
        assert np.array_equal(outs["on"][0][d], ref[d])


@pytest.mark.parametrize("tile", ["auto", "single"])
def test_split_gemm_rs_random_within_tolerance(dev, tile):
    outs, ref = run_rs(dev, 4, 1024, 448, 2560, mode="randn", tile_config=tile, seed=5)
    assert outs["on"][1] > 0
    for d in range(4):
        _close(outs["on"][0][d], ref[d])
        _close(outs["on"][0][d], outs["off"][0][d])


@pytest.mark.parametrize("mode", ["int", "randn"])
def test_split_gemm_rs_bf16_output(dev, mode):
    outs, ref = run_rs(dev, 4, 1024, 256, 1280, mode=mode, out_dtype="bf16", seed=2)
    assert outs["on"][1] > 0
    for d in range(4):
        want = oracle.round_bf16(ref[d])
        if mode == "int":
            assert np.array_equal(outs["on"][0][d], want)
        else:
            _close(outs["on"][0][d], want)


def test_split_gemm_ar_integer_bit_exact(dev):
    R, M, K, N = 4, 1024, 256, 1280
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=4)
    plan = B.fo_plan("gemm_ar", R, M, N, K * R, tail_split="on")
    Y = [torch.empty(M, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_ar(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y, ws)
    _status_ok(plan, ws)
    assert B.fo_plan_last_split_tiles(plan) > 0
    ref = oracle.gemm_ar([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for q in range(R):
        assert np.array_equal(_np(Y[q]), ref[q])


# 80 pair tiles (N_r = 1280: G by movers); 128 pair tiles (N_r = 1024: G from the loaded stages)
@pytest.mark.parametrize("M,N", [(1024, 5120), (2048, 4096)])
@pytest.mark.parametrize("transport", ["peer_read", "copy"])
@pytest.mark.parametrize("mode", ["int", "randn"])
def test_split_ag_gemm(dev, transport, mode, M, N):
    R, K = 4, 320
    inp = ag_gemm_inputs(R, M, K, N // R, mode=mode, seed=1)
    plan = B.fo_plan("ag_gemm", R, M, N, K, ag_transport=transport, tail_split="on")
    bufs, Y = _guarded(R, (M, N // R), torch.bfloat16, dev)
    G = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_ag_gemm(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y, G, ws)
        _status_ok(plan, ws)
    _guards_intact(bufs)
    assert B.fo_plan_last_split_tiles(plan) > 0
    ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for r in range(R):
        want = oracle.round_bf16(ref[r])
        if mode == "int":
            assert np.array_equal(_np(Y[r]), want)
        else:
            _close(_np(Y[r]), want)
        assert np.array_equal(_np(G[r]), gathered)


def test_split_dp_grad_rs_integer_bit_exact(dev):
    R, T, M, N = 4, 256, 1024, 1280           # 80 pair tiles
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=3)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, tail_split="on")
    dW = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW, ws)
    _status_ok(plan, ws)
    assert B.fo_plan_last_split_tiles(plan) > 0
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        assert np.array_equal(_np(dW[d]), ref[d])


def test_full_size_ag_gemm_qkv_is_split_and_within_tolerance(dev):
    from ag_gemm_gb300.inputs import WORKLOADS
    w = WORKLOADS["ag_gemm_qkv_r4_s4096_h4096_n3072"]
    R, M, K, Nr = w.R, w.dims["M"], w.dims["K"], w.dims["N"]
    inp = w.make()
    plan = B.fo_plan("ag_gemm", R, M, Nr * R, K)
    Y = [torch.empty(M, Nr, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_ag_gemm(plan, [x.to(dev) for x in inp["X"]], [x.to(dev) for x in inp["W"]], Y, None, ws)
    _status_ok(plan, ws)
    assert B.fo_plan_last_split_tiles(plan) == 160     # 8 tiles past 10 waves of 76 pairs, plus two waves
    Xn = [_np(x) for x in inp["X"]]
    Wn = [_np(x) for x in inp["W"]]
    rng = np.random.default_rng(9)
    for r in range(R):
        rows = np.sort(np.concatenate([rng.choice(M, 40, replace=False), [M - 1, M - 2]]))
        _close(_np(Y[r][torch.as_tensor(rows, device=dev)]), oracle.round_bf16(oracle.ag_gemm_rows(Xn, Wn, r, rows)))


def test_auto_cuts_only_long_all_gather_tiles(dev):
    # AUTO leaves reduce-scatter plans and short or single-wave launches whole.
    R, M, K, N = 4, 1024, 256, 1280
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=0)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_rs(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y, ws)
    _status_ok(plan, ws)
    assert B.fo_plan_last_split_tiles(plan) == 0
