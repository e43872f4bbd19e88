"""GPU parity of the ring reduce-scatter (FO_RS_RING) against the CPU oracle.

Under the ring, each hop of chunk c's chain adds its partial to the running
sum its ring predecessor forwarded, and forwards the result; the owner is
last. Integer-valued inputs must match the oracle bit for bit (the plain
collective and the oracle's literal ring simulation agree there). The ring
adds in step order, and so does the direct algorithm's deterministic mode
under the same kernel order, so with random inputs the two must agree bit
for bit as well.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import WORKLOADS, dp_grad_inputs, gemm_rs_inputs

pytestmark = pytest.mark.gpu

FRO_TOL = 1e-3
MAX_TOL = 2e-2
GUARD = 64
CANARY = -7.0e33
TILES = ["auto", "single"]


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


def _assert_close(got, ref):
    fro, mx, _ = oracle.rel_errors(got, ref)
    assert fro <= FRO_TOL and mx <= MAX_TOL, f"rel fro {fro:.3e}, max rel {mx:.3e}"


def run_rs(dev, R, M, K, N, *, rs_algo="ring", dtype="bf16", mode="int", layout="kn", seed=0, tile="auto",
           interleave="auto", out_dtype="f32", deterministic=False, repeat=1, inject="none", timeout_ns=0):
    inp = gemm_rs_inputs(R, M, K, N, dtype=dtype, mode=mode, seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, in_dtype=dtype, out_dtype=out_dtype, w_layout=layout,
                     tile_config=tile, interleave=interleave, rs_algo=rs_algo, deterministic=deterministic,
                     fault_inject=inject, timeout_ns=timeout_ns)
    X = [x.to(dev) for x in inp["X"]]
    W = [(w if layout == "kn" else w.t().contiguous()).to(dev) for w in inp["W"]]
    bufs, Y = _guarded(R, (M // R, N), torch.float32 if out_dtype == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    outs = []
    for _ in range(repeat):
        B.fo_gemm_rs(plan, X, W, Y, ws)
        if inject != "none":
            return plan, ws, inp, X, W, Y
        _status_ok(plan, ws)
        outs.append([_np(y) for y in Y])
    _guards_intact(bufs)
    return outs, inp


def _ref(inp):
    return oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("interleave", ["auto", "lockstep", "skewed"])
@pytest.mark.parametrize("R,M,K,N,layout", [
    (2, 256, 512, 512, "kn"),      # two ranks, whole tiles
    (4, 800, 200, 328, "kn"),      # ragged rows per chunk, K and N
    (8, 2048, 64, 256, "nk"),      # eight ranks, one k-block
    (3, 600, 136, 264, "nk"),      # odd R
])
def test_ring_rs_integer_bit_exact(dev, R, M, K, N, layout, tile, interleave):
    outs, inp = run_rs(dev, R, M, K, N, layout=layout, tile=tile, interleave=interleave)
    ref = _ref(inp)
    sim = oracle.simulate_gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]], ring=True)
    for d in range(R):
        assert np.array_equal(outs[0][d], ref[d]), f"shard {d}"
        assert np.array_equal(sim[d], ref[d])


def test_ring_rs_one_rank_is_a_plain_gemm(dev):
    outs, inp = run_rs(dev, 1, 256, 512, 512)
    assert np.array_equal(outs[0][0], _ref(inp)[0])


def test_ring_rs_fp32_inputs_tf32_bit_exact(dev):
    outs, inp = run_rs(dev, 2, 256, 512, 512, dtype="f32", layout="nk")
    ref = _ref(inp)
    for d in range(2):
        assert np.array_equal(outs[0][d], ref[d])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("interleave", ["lockstep", "skewed"])
def test_ring_equals_in_order_direct_adds_bitwise(dev, tile, interleave):
    # Random inputs: the ring's additions (hop order) and the direct
    # algorithm's deterministic additions (kernel order) are the same fp32
    # additions in the same order.
    R, M, K, N = 4, 1024, 384, 520
    ring, inp = run_rs(dev, R, M, K, N, mode="randn", tile=tile, interleave=interleave, seed=7)
    direct, _ = run_rs(dev, R, M, K, N, rs_algo="direct", deterministic=True, mode="randn", tile=tile,
                       interleave=interleave, seed=7)
    ref = _ref(inp)
    for d in range(R):
        assert np.array_equal(ring[0][d], direct[0][d]), f"shard {d}"
        _assert_close(ring[0][d], ref[d])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("mode", ["int", "randn"])
def test_ring_rs_bf16_output_is_rounded_once(dev, tile, mode):
    R, M, K, N = 4, 800, 200, 328
    outs, inp = run_rs(dev, R, M, K, N, mode=mode, tile=tile, out_dtype="bf16", seed=3)
    ref = _ref(inp)
    for d in range(R):
        want = oracle.round_bf16(ref[d])
        if mode == "int":
            assert np.array_equal(outs[0][d], want)
        else:
            _assert_close(outs[0][d], want)


def test_ring_rs_repeated_calls_reuse_workspace(dev):
    outs, inp = run_rs(dev, 4, 1024, 256, 512, repeat=3)
    ref = _ref(inp)
    for rep in outs:
        for d in range(4):
            assert np.array_equal(rep[d], ref[d])


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("R,T,M,N", [(2, 256, 256, 256), (4, 200, 800, 328), (8, 128, 1024, 256)])
def test_ring_dp_grad_rs_integer_bit_exact(dev, R, T, M, N, tile):
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=3)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, tile_config=tile, rs_algo="ring")
    bufs, dW = _guarded(R, (M // R, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW, ws)
    _status_ok(plan, ws)
    _guards_intact(bufs)
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        assert np.array_equal(_np(dW[d]), ref[d]), f"shard {d}"


def test_ring_missing_forward_times_out_and_workspace_recovers(dev):
    # The first hop of chunk 0 (rank 1 at step 0) does not release its
    # forward: the second hop (rank 0 at step 1, the owner) must time out.
    R, M, K, N = 2, 256, 128, 256
    plan, ws, inp, X, W, Y = run_rs(dev, R, M, K, N, inject="skip_signal", timeout_ns=20_000_000)
    code, info = B.fo_status_query(plan, ws)
    assert code == B.FO_ERR_TIMEOUT
    assert info == [B.FO_ERR_TIMEOUT, 0, 1, 0]
    good = B.fo_plan("gemm_rs", R, M, N, K * R, rs_algo="ring")
    B.fo_gemm_rs(good, X, W, Y, ws)
    _status_ok(good, ws)
    ref = _ref(inp)
    for d in range(R):
        assert np.array_equal(_np(Y[d]), ref[d])


def test_full_size_ring_gemm_rs_down_proj(dev):
    w = WORKLOADS["gemm_rs_down_r8_t8192_k1792_n4096"]
    R, M, K, N = w.R, w.dims["M"], w.dims["K"], w.dims["N"]
    inp = w.make()
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, rs_algo="ring")
    X = [x.to(dev) for x in inp["X"]]
    W = [x.to(dev) for x in inp["W"]]
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_rs(plan, X, W, Y, ws)
    _status_ok(plan, ws)
    Xn = [_np(x) for x in inp["X"]]
    Wn = [_np(x) for x in inp["W"]]
    rng = np.random.default_rng(2)
    for d in range(R):
        rows = rng.choice(M // R, size=48, replace=False)
        rows[:2] = [0, M // R - 1]
        rows = np.sort(rows)
        _assert_close(_np(Y[d][torch.as_tensor(rows, device=dev)]), oracle.gemm_rs_rows(Xn, Wn, d, rows))
