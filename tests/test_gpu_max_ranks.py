"""GPU parity at the largest rank count a plan accepts (R = 16): every op (the
all-to-all included), a ragged case, both tile configurations, the bf16
output, the ring reduce-scatter and both all-gather transports with gather
buffers. Integer
inputs, so every result must match the oracle bit for bit; guard bands
around every output catch stray writes.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import gemm_rs_inputs
from test_gpu_parity import Guarded, _np, _status_ok, _ws, run_ag, run_ag_gather, run_dp, run_gemm_rs

pytestmark = pytest.mark.gpu

R = 16


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


@pytest.mark.parametrize("tile", ["auto", "single"])
@pytest.mark.parametrize("M,K,N,layout", [
    (4096, 64, 256, "kn"),       # 256-row chunks
    (1616, 72, 200, "nk"),       # ragged: 101 rows per chunk, N 200
])
def test_gemm_rs_sixteen_ranks(dev, tile, M, K, N, layout):
    outs, ref = run_gemm_rs(dev, R, M, K, N, w_layout=layout, tile=tile)
    for d in range(R):
        assert np.array_equal(outs[0][d], ref[d]), f"shard {d}"


@pytest.mark.parametrize("rs_algo,out_dtype", [("direct", "bf16"), ("ring", "f32"), ("ring", "bf16")])
def test_gemm_rs_sixteen_ranks_bf16_and_ring(dev, rs_algo, out_dtype):
    M, K, N = 2048, 64, 264
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=7)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, rs_algo=rs_algo, out_dtype=out_dtype)
    Y = Guarded(R, (M // R, N), torch.float32 if out_dtype == "f32" else torch.bfloat16, dev)
    ws = _ws(plan, dev)
    for _ in range(2):
        B.fo_gemm_rs(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
        _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        want = ref[d] if out_dtype == "f32" else oracle.round_bf16(ref[d])
        assert np.array_equal(_np(Y.views[d]), want), f"shard {d}"


def test_gemm_ar_sixteen_ranks(dev):
    M, K, N = 2048, 64, 256
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=8)
    plan = B.fo_plan("gemm_ar", R, M, N, K * R)
    Y = Guarded(R, (M, N), torch.float32, dev)
    ws = _ws(plan, dev)
    B.fo_gemm_ar(plan, [x.to(dev) for x in inp["X"]], [w.to(dev) for w in inp["W"]], Y.views, ws)
    _status_ok(plan, ws)
    Y.check()
    ref = oracle.gemm_ar([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for q in range(R):
        assert np.array_equal(_np(Y.views[q]), ref[q]), f"rank {q}"


@pytest.mark.parametrize("tile", ["auto", "single"])
@pytest.mark.parametrize("M,K,N,layout", [
    (4096, 128, 4096, "kn"),     # 256-row shards, 256 columns per rank
    (1600, 72, 1664, "nk"),      # ragged: 100-row shards, 104 columns per rank
])
def test_ag_gemm_sixteen_ranks(dev, tile, M, K, N, layout):
    got, ref = run_ag(dev, R, M, K, N, layout=layout, tile=tile)
    for r in range(R):
        assert np.array_equal(got[r], oracle.round_bf16(ref[r])), f"rank {r}"


@pytest.mark.parametrize("transport,N", [
    ("peer_read", 4096),         # 256 columns per rank: gather output from the loaded stages
    ("peer_read", 20480),        # 1280 columns per rank: gather output by mover warps
    ("copy", 4096),              # ring-forwarded shards, lockstep order
])
def test_ag_gemm_sixteen_ranks_gather_buffers(dev, transport, N):
    M, K = 2048, 64
    for code, info, Y, G, inp in run_ag_gather(dev, R, M, K, N, transport=transport, seeds=(1, 2)):
        assert code == 0, info
        ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for r in range(R):
            assert np.array_equal(Y[r], oracle.round_bf16(ref[r])), f"rank {r}"
            assert np.array_equal(G[r], gathered), f"gather buffer {r}"


@pytest.mark.parametrize("tile", ["auto", "single"])
def test_dp_grad_rs_sixteen_ranks(dev, tile):
    got, ref = run_dp(dev, R, 128, 4096, 256, tile=tile)
    for d in range(R):
        assert np.array_equal(got[d], ref[d]), f"shard {d}"


@pytest.mark.parametrize("tile", ["auto", "single"])
@pytest.mark.parametrize("M,K,N,layout", [
    (4096, 128, 4096, "kn"),     # 256 tokens per rank, blocks of 256 columns
    (1600, 72, 1664, "nk"),      # ragged: 100 tokens per rank, blocks of 104 columns
])
def test_a2a_sixteen_ranks(dev, tile, M, K, N, layout):
    from test_gpu_a2a import run_a2a
    outs, ref, _ = run_a2a(dev, R, M, K, N, layout=layout, tile=tile)
    for c in range(R):
        assert np.array_equal(outs[0][c], oracle.round_bf16(ref[c])), f"rank {c}"
