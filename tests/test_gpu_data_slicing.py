"""The data-slicing baseline that bench.py sweeps over chunk counts computes
the same sums as the reduce-scatter: for each slice j of M/S rows, rank d
holds its M/(S*R) rows of sum_r X_r[slice j] . W_r, slices in order.
Integer-valued inputs keep every fp32 sum exact, so the check is bit for bit.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import gemm_rs_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _np(t):
    return t.detach().to("cpu").double().numpy()


@pytest.mark.parametrize("R,M,K,N,S", [
    (4, 2048, 256, 512, 1),     # one slice: the serial unfused path
    (4, 2048, 256, 512, 2),     # 256-row chunks: CTA-pair tiles
    (4, 2048, 256, 512, 4),     # 128-row chunks: single-CTA tiles
    (8, 2048, 192, 640, 8),     # 32-row chunks: ragged single-CTA tiles
])
def test_data_slicing_matches_the_sliced_sums(dev, R, M, K, N, S):
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=S)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]
    Y = [torch.full((M // R, N), -1.0, device=dev) for _ in range(R)]
    ds = bench.DataSlicing(B, R, M, N, K, S, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):                       # the second call reuses the partial buffers
        ds(X, W, Y, stream)
    torch.cuda.synchronize()
    Ms = M // S
    Xn = [_np(x) for x in inp["X"]]
    Wn = [_np(w) for w in inp["W"]]
    want = [[] for _ in range(R)]
    for j in range(S):
        shards = oracle.gemm_rs([x[j * Ms:(j + 1) * Ms] for x in Xn], Wn)
        for d in range(R):
            want[d].append(shards[d])
    for d in range(R):
        assert np.array_equal(_np(Y[d]), np.concatenate(want[d])), f"rank {d}"
