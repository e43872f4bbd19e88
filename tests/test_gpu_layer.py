"""The projections of one TP-SP transformer layer, forward and backward,
through the fused collectives (ag_gemm_gb300.layer): every output against the
CPU oracle. Integer inputs make every fp32 sum exact, so fp32 outputs match
bit for bit and bf16 outputs match the oracle rounded once to bf16."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _np(t):
    return t.detach().to("cpu").double().numpy()


def _T(ws):
    return [w.T for w in ws]


@pytest.fixture(scope="module", params=[False, True], ids=["shards_in_place", "keep_gathered"])
def layer(request):
    import __graft_entry__
    __graft_entry__.build()
    from ag_gemm_gb300.layer import LayerShape, TpspLayerProjections
    L = TpspLayerProjections(LayerShape(R=4, T=256, H=128, F=256), device="cuda:0", mode="int", seed=9,
                             keep_gathered=request.param)
    L.forward()
    L.backward()
    torch.cuda.synchronize()
    assert L.status() == [0] * len(L.plans)
    assert L.launches == 12
    return L


def test_forward_projections(layer):
    L = layer
    R = L.s.R
    x, attn, act = [_np(t) for t in L.x], [_np(t) for t in L.attn], [_np(t) for t in L.act]
    Wqkv, Wo, Wug, Wd = ([_np(t) for t in W] for W in (L.Wqkv, L.Wo, L.Wug, L.Wd))
    y_qkv, Gx = oracle.ag_gemm(x, Wqkv)
    h = oracle.gemm_rs(attn, Wo)
    y = oracle.gemm_rs(act, Wd)
    for r in range(R):
        assert np.array_equal(_np(L.y_qkv[r]), oracle.round_bf16(y_qkv[r]))
        if L.keep_gathered:
            assert np.array_equal(_np(L.Gx[r]), Gx)
        assert np.array_equal(_np(L.h[r]), oracle.round_bf16(h[r]))
        assert np.array_equal(_np(L.y[r]), oracle.round_bf16(y[r]))
    h_gpu = [_np(t) for t in L.h]          # bf16 h as produced feeds up|gate
    y_ug, Gh = oracle.ag_gemm(h_gpu, Wug)
    for r in range(R):
        assert np.array_equal(_np(L.y_ug[r]), oracle.round_bf16(y_ug[r]))
        if L.keep_gathered:
            assert np.array_equal(_np(L.Gh[r]), Gh)


def test_backward_projections(layer):
    L = layer
    R = L.s.R
    np_ = lambda ts: [_np(t) for t in ts]
    dy, dh, dug, dqkv = np_(L.dy), np_(L.dh), np_(L.dug), np_(L.dqkv)
    Wqkv, Wo, Wug, Wd = np_(L.Wqkv), np_(L.Wo), np_(L.Wug), np_(L.Wd)
    act, attn = np_(L.act), np_(L.attn)
    Gx, Gh = oracle.all_gather_rows(np_(L.x)), oracle.all_gather_rows(np_(L.h))   # h as produced
    d_act, G_dy = oracle.ag_gemm(dy, _T(Wd))
    d_attn, G_dh = oracle.ag_gemm(dh, _T(Wo))
    d_h = oracle.gemm_rs(dug, _T(Wug))
    d_x = oracle.gemm_rs(dqkv, _T(Wqkv))
    dWd = oracle.weight_grads(act, [G_dy] * R)
    dWo = oracle.weight_grads(attn, [G_dh] * R)
    dWug = oracle.weight_grads([Gh] * R, dug)
    dWqkv = oracle.weight_grads([Gx] * R, dqkv)
    for r in range(R):
        assert np.array_equal(_np(L.d_act[r]), oracle.round_bf16(d_act[r]))
        assert np.array_equal(_np(L.d_attn[r]), oracle.round_bf16(d_attn[r]))
        if L.keep_gathered:
            assert np.array_equal(_np(L.G_dy[r]), G_dy)
            assert np.array_equal(_np(L.G_dh[r]), G_dh)
        assert np.array_equal(_np(L.d_h_from_ug[r]), oracle.round_bf16(d_h[r]))
        assert np.array_equal(_np(L.d_x[r]), oracle.round_bf16(d_x[r]))
        assert np.array_equal(_np(L.dWd[r]), dWd[r].T)      # row-parallel grads in [out x in]
        assert np.array_equal(_np(L.dWo[r]), dWo[r].T)
        assert np.array_equal(_np(L.dWug[r]), dWug[r])
        assert np.array_equal(_np(L.dWqkv[r]), dWqkv[r])
