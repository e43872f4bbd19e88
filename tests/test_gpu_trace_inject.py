"""GPU tests of the launch trace (per-CTA %globaltimer stamps) and of the
delay hook that holds the first chunk task of a launch.

A delay below the wait bound must leave every result bit-exact: the tiles
that depend on the delayed task's partials (RS/DP) or tiles (AG) have to
wait for them, whatever the reduce-scatter algorithm, schedule or
transport. A delay beyond the bound must surface as FO_ERR_TIMEOUT through
fo_status_query, after which the workspace serves a healthy plan again.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import ag_gemm_inputs, dp_grad_inputs, gemm_rs_inputs

pytestmark = pytest.mark.gpu

DELAY_US = 300


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _np(t):
    return t.detach().to("cpu").double().numpy()


def _ws(plan, dev):
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)
    return ws


def _rs(dev, R=4, M=1024, K=256, N=512, seed=0, **kw):
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=seed)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, **kw)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]
    Y = [torch.full((M // R, N), -1.0, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_gemm_rs(plan, X, W, Y, ws)
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    return plan, ws, X, W, Y, ref


@pytest.mark.parametrize("tile", ["auto", "single"])
def test_trace_stamps_are_ordered_and_show_the_tail(dev, tile):
    plan, ws, X, W, Y, ref = _rs(dev, trace=True, tile_config=tile)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, info
    for d in range(4):
        assert np.array_equal(_np(Y[d]), ref[d])
    rows = B.fo_trace_query(plan, ws)
    assert 0 < len(rows) <= torch.cuda.get_device_properties(0).multi_processor_count
    leaders = [r for r in rows if r[1]]
    assert leaders and len(leaders) == (len(rows) // 2 if tile == "auto" else len(rows))
    for r in rows:
        assert r[0] > 0 and r[7] == 0
        assert all(r[0] <= r[k] <= r[6] for k in (2, 3, 4, 5))
        if r[1]:
            assert r[0] < r[1] <= r[6]
    s = B.trace_summary(rows)
    assert 0 <= s["exposed_tail_ns"] < s["span_ns"] < 1_000_000_000
    assert 0 < s["mma_end_ns"] <= s["span_ns"] and s["transfers_end_ns"] <= s["span_ns"]


def test_trace_follows_every_launch(dev):
    plan, ws, X, W, Y, ref = _rs(dev, trace=True)
    first = B.fo_trace_query(plan, ws)
    B.fo_gemm_rs(plan, X, W, Y, ws)
    second = B.fo_trace_query(plan, ws)
    assert min(r[0] for r in second) > max(r[6] for r in first)


@pytest.mark.parametrize("kw", [
    dict(),                                              # direct, skewed
    dict(deterministic=True),                            # direct, adds in step order
    dict(interleave="lockstep"),
    dict(rs_algo="ring"),
    dict(tile_config="single"),
])
def test_delayed_first_task_keeps_gemm_rs_exact(dev, kw):
    plan, ws, X, W, Y, ref = _rs(dev, fault_inject="delay_first_task", inject_delay_us=DELAY_US, trace=True, **kw)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, info
    for d in range(4):
        assert np.array_equal(_np(Y[d]), ref[d]), f"shard {d}"
    assert B.trace_summary(B.fo_trace_query(plan, ws))["span_ns"] >= DELAY_US * 1000


def test_delayed_first_task_keeps_dp_grad_rs_exact(dev):
    R, T, M, N = 4, 256, 1024, 512
    inp = dp_grad_inputs(R, T, M, N, mode="int", seed=3)
    plan = B.fo_plan("dp_grad_rs", R, M, N, T, fault_inject="delay_first_task", inject_delay_us=DELAY_US)
    dW = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_dp_grad_rs(plan, [x.to(dev) for x in inp["X"]], [y.to(dev) for y in inp["dY"]], dW, ws)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, info
    ref = oracle.dp_grad_rs([_np(x) for x in inp["X"]], [_np(y) for y in inp["dY"]])
    for d in range(R):
        assert np.array_equal(_np(dW[d]), ref[d])


@pytest.mark.parametrize("transport", ["peer_read", "copy"])
def test_delayed_first_task_keeps_ag_gemm_exact(dev, transport):
    R, M, K, N = 4, 1024, 256, 512
    inp = ag_gemm_inputs(R, M, K, N // R, mode="int", seed=1)
    plan = B.fo_plan("ag_gemm", R, M, N, K, ag_transport=transport, fault_inject="delay_first_task",
                     inject_delay_us=DELAY_US)
    Y = [torch.empty(M, N // R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    G = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    ws = _ws(plan, dev)
    B.fo_ag_gemm(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y, G, ws)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, info
    ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for r in range(R):
        assert np.array_equal(_np(Y[r]), oracle.round_bf16(ref[r]))
        assert np.array_equal(_np(G[r]), gathered)


def test_delay_beyond_the_wait_bound_times_out_and_recovers(dev):
    # The first task holds for 200 ms; tiles waiting for its partials give up
    # after 20 ms and the launch reports the timeout.
    plan, ws, X, W, Y, ref = _rs(dev, fault_inject="delay_first_task", inject_delay_us=200_000,
                                 timeout_ns=20_000_000)
    code, info = B.fo_status_query(plan, ws)
    assert code == B.FO_ERR_TIMEOUT
    assert info[0] == B.FO_ERR_TIMEOUT
    good = B.fo_plan("gemm_rs", 4, 1024, 512, 256 * 4)
    B.fo_gemm_rs(good, X, W, Y, ws)
    code, info = B.fo_status_query(good, ws)
    assert code == 0, info
    for d in range(4):
        assert np.array_equal(_np(Y[d]), ref[d])
