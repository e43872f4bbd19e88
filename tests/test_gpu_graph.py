"""The fused calls (the attention call, the weight gradient over token shards
and a whole layer step) captured in a CUDA graph and replayed.

A call leaves its workspace ready for the next one (readiness counters reset
themselves, the all-gather flags carry a launch epoch), so a captured call
can be replayed with new contents in the same input buffers. Each replay must
match the oracle bit for bit in the integer mode.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import ag_gemm_inputs, dp_grad_inputs, gemm_rs_inputs

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("tile,dtype", [("auto", "bf16"), ("single", "bf16"), ("auto", "f32")])
def test_gemm_rs_replays_from_a_cuda_graph(dev, tile, dtype):
    # (fp32 inputs with W as [K x N]: the graph holds the transpose of W into
    # the workspace and the fused launch.)
    R, M, K, N = 4, 1024, 256, 512
    plan = B.fo_plan("gemm_rs", R, M, N, K * R, tile_config=tile, in_dtype=dtype)
    ws = _ws(plan, dev)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    X = [torch.empty(M, K, dtype=tdt, device=dev) for _ in range(R)]
    W = [torch.empty(K, N, dtype=tdt, device=dev) for _ in range(R)]
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    for t in X + W:
        t.zero_()
    B.fo_gemm_rs(plan, X, W, Y, ws)          # first call outside the capture: device set-up, encodings
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fo_gemm_rs(plan, X, W, Y, ws)
    for seed in (1, 2, 3):
        inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=seed, dtype=dtype)
        for r in range(R):
            X[r].copy_(inp["X"][r])
            W[r].copy_(inp["W"][r])
        g.replay()
        torch.cuda.synchronize()
        code, info = B.fo_status_query(plan, ws)
        assert code == 0, info
        ref = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for d in range(R):
            assert np.array_equal(_np(Y[d]), ref[d]), f"seed {seed} shard {d}"


@pytest.mark.parametrize("transport", ["peer_read", "copy"])
def test_ag_gemm_replays_from_a_cuda_graph(dev, transport):
    R, M, K, N = 4, 1024, 256, 512
    plan = B.fo_plan("ag_gemm", R, M, N, K, ag_transport=transport)
    ws = _ws(plan, dev)
    X = [torch.zeros(M // R, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    W = [torch.zeros(K, N // R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Y = [torch.empty(M, N // R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    G = [torch.empty(M, K, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    B.fo_ag_gemm(plan, X, W, Y, G, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fo_ag_gemm(plan, X, W, Y, G, ws)
    for seed in (1, 2, 3):
        inp = ag_gemm_inputs(R, M, K, N // R, mode="int", seed=seed)
        for r in range(R):
            X[r].copy_(inp["X"][r])
            W[r].copy_(inp["W"][r])
        g.replay()
        torch.cuda.synchronize()
        code, info = B.fo_status_query(plan, ws)
        assert code == 0, info
        ref, gathered = oracle.ag_gemm([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
        for r in range(R):
            assert np.array_equal(_np(Y[r]), oracle.round_bf16(ref[r])), f"seed {seed} rank {r}"
            assert np.array_equal(_np(G[r]), gathered)


@pytest.mark.parametrize("causal", [False, True])
def test_attn_rs_replays_from_a_cuda_graph(dev, causal):
    # The attention launch deals its items from a counter in the workspace
    # header that its last CTA sets back to zero, so a captured call can be
    # replayed. Each replay's O must equal a direct call's bit for bit (each
    # output tile comes from one CTA in a fixed order), and Y must match the
    # oracle's reduce-scatter of that O.
    R, T, heads, H, D = 2, 512, 2, 256, 128
    plan = B.fo_plan("gemm_rs", R, T, H, R * heads * D)
    ws = _ws(plan, dev)
    bf = torch.bfloat16
    Q, K, V = ([torch.zeros(T, heads * D, dtype=bf, device=dev) for _ in range(R)] for _ in range(3))
    Wo = [torch.zeros(heads * D, H, dtype=bf, device=dev) for _ in range(R)]
    O = [torch.empty(T, heads * D, dtype=bf, device=dev) for _ in range(R)]
    Y = [torch.empty(T // R, H, device=dev) for _ in range(R)]
    B.fo_attn_rs(plan, Q, K, V, Wo, O, Y, heads, causal, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fo_attn_rs(plan, Q, K, V, Wo, O, Y, heads, causal, ws)
    O2 = [torch.empty_like(o) for o in O]
    Y2 = [torch.empty_like(y) for y in Y]
    for seed in (1, 2, 3):
        gen = torch.Generator().manual_seed(seed)
        for r in range(R):
            for t in (Q[r], K[r], V[r]):
                t.copy_(torch.randn(t.shape, generator=gen).to(bf))
            Wo[r].copy_((torch.randn(Wo[r].shape, generator=gen) * 0.02).to(bf))
        g.replay()
        torch.cuda.synchronize()
        code, info = B.fo_status_query(plan, ws)
        assert code == 0, info
        B.fo_attn_rs(plan, Q, K, V, Wo, O2, Y2, heads, causal, ws)
        torch.cuda.synchronize()
        assert B.fo_status_query(plan, ws)[0] == 0
        for r in range(R):
            assert torch.equal(O[r], O2[r]), f"seed {seed} rank {r}"
        ref = oracle.gemm_rs([_np(o) for o in O], [_np(w) for w in Wo])
        for d in range(R):
            fro, mx, _ = oracle.rel_errors(_np(Y[d]), ref[d])
            assert fro <= 1e-3 and mx <= 2e-2, f"seed {seed} shard {d}: {fro:.2e} {mx:.2e}"


@pytest.mark.parametrize("placement", ["separate", "back_to_back", "spaced"])
def test_partials_sharded_replays_from_a_cuda_graph(dev, placement):
    from test_gpu_parity import _place_shards
    R, T, M, N = 4, 512, 256, 192
    plan = B.fo_plan("dp_grad_rs", R, M, N, T)
    ws = _ws(plan, dev)
    bf = torch.bfloat16
    A = _place_shards([torch.zeros(T // R, M, dtype=bf) for _ in range(R)], placement, dev)
    dY = [torch.zeros(T, N, dtype=bf, device=dev) for _ in range(R)]
    P = [torch.empty(M, N, device=dev) for _ in range(R)]
    B.fo_gemm_partials_sharded(plan, A, dY, P, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.fo_gemm_partials_sharded(plan, A, dY, P, ws)
    for seed in (1, 2, 3):
        inp = dp_grad_inputs(R, T, M, N, mode="int", seed=seed)
        for s_, a in zip(inp["X"][0].split(T // R), A):
            a.copy_(s_)
        for r in range(R):
            dY[r].copy_(inp["dY"][r])
        g.replay()
        torch.cuda.synchronize()
        code, info = B.fo_status_query(plan, ws)
        assert code == 0, info
        ref = oracle.weight_grads([oracle.all_gather_rows([_np(a) for a in A])] * R, [_np(y) for y in dY])
        for r in range(R):
            assert np.array_equal(_np(P[r]), ref[r]), f"seed {seed} rank {r}"


def test_layer_step_replays_from_a_cuda_graph(dev):
    # One forward + backward of the TP-SP layer (12 launches) captured once;
    # every replay on fresh inputs equals an eager step bit for bit.
    from ag_gemm_gb300.layer import LayerShape, TpspLayerProjections
    L = TpspLayerProjections(LayerShape(R=4, T=512, H=256, F=512), device=dev, mode="int", seed=3)
    L.forward()
    L.backward()
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.forward(s)
        L.backward(s)
    outs = lambda: [t.clone() for ts in (L.y_qkv, L.h, L.y_ug, L.y, L.d_act, L.dWd, L.d_h_from_ug, L.dWug,
                                          L.d_attn, L.dWo, L.d_x, L.dWqkv) for t in ts]
    gen = torch.Generator().manual_seed(11)
    for _ in range(2):
        for ts in (L.x, L.attn, L.act, L.dy, L.dh, L.dug, L.dqkv):
            for t in ts:
                t.copy_(torch.randint(-4, 5, t.shape, generator=gen).to(t.dtype))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        got = outs()
        L.forward()
        L.backward()
        torch.cuda.synchronize()
        assert L.status() == [0] * len(L.plans)
        for a, b in zip(got, outs()):
            assert torch.equal(a, b)
