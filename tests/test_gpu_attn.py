"""GPU parity of query-split attention with its row-parallel output
projection (fo_attn_rs, and its attention launch alone, fo_attention)
against the CPU oracle, through the C ABI.

Tolerances. The tensor cores take the softmax weights in bf16 (8
significant bits, unit roundoff u = 2^-8), each weight e_k / l with a
relative error of at most u, so element (i, j) of O moves by at most
u * sum_k p_ik |v_kj|: the attention of |V|, which the oracle computes.
O is then rounded once to bf16 on both sides; values that round apart
differ by at most one bf16 step, 2^-7 |O_ij|. Elementwise, O is held to
1.25 (u * attention(|V|) + 2^-7 |O|); the fp32 score, exponent and sum
errors fit in the quarter of slack. In Frobenius norm O is held to 4e-3
of the reference. The projection is checked separately at the stated GEMM
tolerances (relative Frobenius 1e-3, elementwise 2e-2) against the
oracle's reduce-scatter of the O the GPU produced; end to end, Y is held
to the same 4e-3 Frobenius bound as O.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B

pytestmark = pytest.mark.gpu

O_FRO = 4e-3
U_BF16 = 2.0 ** -8       # unit roundoff of bf16
ULP_BF16 = 2.0 ** -7     # one bf16 step, relative to the value
O_SLACK = 1.25
FRO_TOL, MAX_TOL = 1e-3, 2e-2
D = 128


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    return torch.device("cuda:0")


def _np(t):
    return t.detach().to("cpu").double().numpy()


def _inputs(R, T, heads, H, seed, q_scale=1.0, growing_keys=False):
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    Q = [(torch.randn(T, heads * D, generator=g) * q_scale).to(bf) for _ in range(R)]
    K = [torch.randn(T, heads * D, generator=g).to(bf) for _ in range(R)]
    V = [torch.randn(T, heads * D, generator=g).to(bf) for _ in range(R)]
    Wo = [(torch.randn(heads * D, H, generator=g) * 0.02).to(bf) for _ in range(R)]
    if growing_keys:
        # Scores that grow along the keys: each row's maximum keeps rising
        # from one 128-key block to the next, so the output must be
        # rescaled again and again.
        ramp = torch.linspace(0.0, 6.0, T)[:, None]
        for r in range(R):
            Q[r] = (torch.ones(T, heads * D) * 0.5).to(bf)
            K[r] = (torch.randn(T, heads * D, generator=g) * 0.1 + ramp).to(bf)
    return Q, K, V, Wo


def run_attn(dev, R, T, heads, H, causal, seed=0, out="f32", **kw):
    Q, K, V, Wo = _inputs(R, T, heads, H, seed, **kw)
    plan = B.fo_plan("gemm_rs", R, T, H, R * heads * D, out_dtype=out)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    dQ, dK, dV, dW = ([t.to(dev) for t in ts] for ts in (Q, K, V, Wo))
    O = [torch.full((T, heads * D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Y = [torch.full((T // R, H), float("nan"), dtype=torch.float32 if out == "f32" else torch.bfloat16,
                    device=dev) for _ in range(R)]
    B.fo_attn_rs(plan, dQ, dK, dV, dW, O, Y, heads, causal, ws)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, f"device status {code} {info}"
    assert B.fo_plan_last_launches(plan) == 2
    return [_np(t) for t in Q], [_np(t) for t in K], [_np(t) for t in V], [_np(t) for t in Wo], \
        [_np(o) for o in O], [_np(y) for y in Y]


def _check_o(got, ref, absw, what):
    """got: the kernel's O; ref: the oracle's O rounded to bf16; absw: the
    oracle's attention of |V| (the per-element weight-rounding bound)."""
    fro = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    bound = O_SLACK * (U_BF16 * absw + ULP_BF16 * np.abs(ref))
    ratio = float(np.max(np.abs(got - ref) / bound))
    assert fro <= O_FRO and ratio <= 1.0, f"{what}: rel fro {fro:.3e}, worst element at {ratio:.2f} of its bound"


def _check_all(Q, K, V, Wo, O, Y, heads, causal, out="f32"):
    R = len(Q)
    for r in range(R):
        ref_o = oracle.round_bf16(oracle.attention(Q[r], K[r], V[r], heads, causal))
        absw = oracle.attention(Q[r], K[r], np.abs(V[r]), heads, causal)
        _check_o(O[r], ref_o, absw, f"O rank {r}")
    # the projection on the O the GPU produced: the GEMM-RS tolerances
    proj = oracle.gemm_rs(O, Wo)
    for d in range(R):
        want = proj[d] if out == "f32" else oracle.round_bf16(proj[d])
        fro, mx, _ = oracle.rel_errors(Y[d], want)
        assert fro <= FRO_TOL and mx <= MAX_TOL, f"Y shard {d}: rel fro {fro:.3e}, max {mx:.3e}"
    # end to end
    ref = oracle.attn_rs(Q, K, V, Wo, heads, causal, round_o=True)
    for d in range(R):
        fro = float(np.linalg.norm(Y[d] - ref[d]) / np.linalg.norm(ref[d]))
        assert fro <= O_FRO, f"Y shard {d} end to end: rel fro {fro:.3e}"


# Query blocks of T/R rows hold (T/R)/128 tiles: one, two, three and four
# tiles per block, R = 1 to 4.
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R,T,heads,H", [(1, 256, 1, 256), (2, 512, 2, 384), (4, 1024, 1, 512),
                                         (2, 256, 1, 256), (2, 768, 2, 256), (3, 1152, 1, 384)])
def test_attn_rs_matches_the_oracle(dev, R, T, heads, H, causal):
    res = run_attn(dev, R, T, heads, H, causal, seed=R * 10 + heads)
    _check_all(*res, heads, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_attn_rs_sharp_scores_and_bf16_output(dev, causal):
    # Queries four times larger: peaked softmax rows; bf16 projection output.
    res = run_attn(dev, 2, 512, 1, 256, causal, seed=7, out="bf16", q_scale=4.0)
    _check_all(*res, 1, causal, out="bf16")


@pytest.mark.parametrize("T", [768, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_attn_rs_growing_maximum_is_rescaled(dev, causal, T):
    res = run_attn(dev, 2, T, 1, 256, causal, seed=8, growing_keys=True)
    _check_all(*res, 1, causal)


def test_attn_rs_repeats_bit_for_bit(dev):
    # Two calls in a row on the same buffers give the same bits.
    R, T, heads, H = 4, 512, 2, 256
    Q, K, V, Wo = _inputs(R, T, heads, H, seed=3)
    plan = B.fo_plan("gemm_rs", R, T, H, R * heads * D)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    dQ, dK, dV, dW = ([t.to(dev) for t in ts] for ts in (Q, K, V, Wo))
    outs = []
    for _ in range(2):
        O = [torch.empty(T, heads * D, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        Y = [torch.empty(T // R, H, device=dev) for _ in range(R)]
        B.fo_attn_rs(plan, dQ, dK, dV, dW, O, Y, heads, True, ws)
        assert B.fo_status_query(plan, ws)[0] == 0
        outs.append(([o.clone() for o in O], [y.clone() for y in Y]))
    for r in range(R):
        assert torch.equal(outs[0][0][r], outs[1][0][r])


def test_attn_rs_llama_shape_sampled(dev):
    # The layer's attention shape: 8192 tokens over R = 8, 4 heads of 128
    # per rank (32 heads), H = 4096, causal; O checked on sampled query rows
    # of every head, Y on sampled rows of every shard.
    R, T, heads, H = 8, 8192, 4, 4096
    Q, K, V, Wo, O, Y = run_attn(dev, R, T, heads, H, True, seed=11)
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([[0, 127, 128, T - 1], rng.choice(T, 12, replace=False)]))
    for r in (0, R - 1):
        Qr = Q[r]
        ref_rows = np.empty((len(rows), heads * D))
        absw = np.empty((len(rows), heads * D))
        for h in range(heads):
            cols = slice(h * D, (h + 1) * D)
            for i, t in enumerate(rows):
                s = (Qr[t, cols] @ K[r][: t + 1, cols].T) / np.sqrt(D)
                w = np.exp(s - s.max())
                ref_rows[i, cols] = (w / w.sum()) @ V[r][: t + 1, cols]
                absw[i, cols] = (w / w.sum()) @ np.abs(V[r][: t + 1, cols])
        _check_o(O[r][rows], oracle.round_bf16(ref_rows), absw, f"O rank {r}")
    srows = np.array([0, 1, 511, 1023])
    for d in range(R):
        want = oracle.gemm_rs_rows(O, Wo, d, srows)
        fro, mx, _ = oracle.rel_errors(Y[d][srows], want)
        assert fro <= FRO_TOL and mx <= MAX_TOL, f"Y shard {d}: rel fro {fro:.3e}, max {mx:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_attention_alone_matches_attn_rs_and_resets_its_counter(dev, causal):
    # fo_attention is the first launch of fo_attn_rs: same O bits, one
    # launch, and the item counter in the workspace header (words 6 and 7)
    # is back at zero when the launch ends, ready for the next one.
    R, T, heads, H = 2, 1024, 2, 256
    Q, K, V, Wo = _inputs(R, T, heads, H, seed=21)
    plan = B.fo_plan("gemm_rs", R, T, H, R * heads * D)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    dQ, dK, dV, dW = ([t.to(dev) for t in ts] for ts in (Q, K, V, Wo))
    O1 = [torch.full((T, heads * D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    O2 = [torch.full((T, heads * D), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Y = [torch.empty(T // R, H, device=dev) for _ in range(R)]
    for _ in range(3):
        B.fo_attention(plan, dQ, dK, dV, O1, heads, causal, ws)
        assert B.fo_plan_last_launches(plan) == 1
        assert B.fo_status_query(plan, ws)[0] == 0
        assert ws[24:32].view(torch.int32).tolist() == [0, 0]
    B.fo_attn_rs(plan, dQ, dK, dV, dW, O2, Y, heads, causal, ws)
    assert B.fo_status_query(plan, ws)[0] == 0
    for r in range(R):
        assert torch.equal(O1[r], O2[r])
        q, k, v = _np(Q[r]), _np(K[r]), _np(V[r])
        ref = oracle.round_bf16(oracle.attention(q, k, v, heads, causal))
        _check_o(_np(O1[r]), ref, oracle.attention(q, k, np.abs(v), heads, causal), f"O rank {r}")


def test_attention_wait_that_runs_out_reports_and_the_next_call_is_exact(dev):
    # One softmax warp of CTA 0 withholds its first "weights written" signal
    # (the plan's skip_signal hook): that CTA's weighted-sum wait runs out
    # (the attention launch's waits give up after 2 s), every role leaves
    # its loops, and the call reports FO_ERR_TIMEOUT. fo_status_query then zeroes the workspace, and
    # a clean call on the same buffers is exact, with the item counter back
    # at zero.
    R, T, heads, H = 2, 1024, 2, 256
    Q, K, V, Wo = _inputs(R, T, heads, H, seed=31)
    bad = B.fo_plan("gemm_rs", R, T, H, R * heads * D, fault_inject="skip_signal")
    good = B.fo_plan("gemm_rs", R, T, H, R * heads * D)
    ws = torch.zeros(max(B.fo_workspace_size(bad), B.fo_workspace_size(good)), dtype=torch.uint8, device=dev)
    dQ, dK, dV = ([t.to(dev) for t in ts] for ts in (Q, K, V))
    O = [torch.empty(T, heads * D, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    B.fo_attention(bad, dQ, dK, dV, O, heads, True, ws)
    code, info = B.fo_status_query(bad, ws)
    assert code == B.FO_ERR_TIMEOUT, (code, info)
    assert ws[24:32].view(torch.int32).tolist() == [0, 0]
    B.fo_attention(good, dQ, dK, dV, O, heads, True, ws)
    assert B.fo_status_query(good, ws)[0] == 0
    assert ws[24:32].view(torch.int32).tolist() == [0, 0]
    for r in range(R):
        q, k, v = _np(Q[r]), _np(K[r]), _np(V[r])
        ref = oracle.round_bf16(oracle.attention(q, k, v, heads, True))
        _check_o(_np(O[r]), ref, oracle.attention(q, k, np.abs(v), heads, True), f"O rank {r}")


@pytest.mark.parametrize("R,T,heads,H,causal", [(16, 2048, 1, 256, True), (16, 4096, 1, 256, False),
                                                (2, 512, 8, 256, True), (8, 2048, 4, 512, False)])
def test_attn_rs_more_ranks_and_heads(dev, R, T, heads, H, causal):
    # The largest rank count (16 query blocks of one tile each, or two),
    # eight heads per rank, and R = 8 without the mask.
    res = run_attn(dev, R, T, heads, H, causal, seed=R + heads)
    _check_all(*res, heads, causal)
