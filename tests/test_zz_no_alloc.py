"""fo_gemm_rs_noalloc: the fused GEMM + reduce-scatter for callers that cannot
allocate device memory (code running inside allocator hooks or host
callbacks, or under a runtime that owns the device memory pool). It keeps its
readiness counters in a static device array instead of a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from ag_gemm_gb300 import binding as B
from ag_gemm_gb300.inputs import gemm_rs_inputs

FRO_TOL = 1e-3
MAX_TOL = 2e-2


def _np(t):
    return t.detach().to("cpu").double().numpy()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    dev = torch.device("cuda:0")
    R, M, K, N = 4, 1000, 200, 328           # ragged: 250 rows per shard, K and N not tile multiples
    inp = gemm_rs_inputs(R, M, K, N, mode="randn", seed=11)
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]

    # The existing entry point, with a workspace.
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)
    Y_ref = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    B.fo_gemm_rs(plan, X, W, Y_ref, ws)
    code, info = B.fo_status_query(plan, ws)
    assert code == 0, info
    ref = [_np(y) for y in Y_ref]

    # The allocation-free entry point, twice in a row into fresh outputs.
    for call in range(2):
        Y = [torch.full((M // R, N), float("nan"), device=dev) for _ in range(R)]
        B.fo_gemm_rs_noalloc(plan, X, W, Y)
        torch.cuda.synchronize()
        for d in range(R):
            fro, mx, _ = oracle.rel_errors(_np(Y[d]), ref[d])
            assert fro <= FRO_TOL and mx <= MAX_TOL, f"call {call} shard {d}: fro {fro:.2e} max {mx:.2e}"
    # And both agree with the CPU oracle.
    want = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for d in range(R):
        fro, mx, _ = oracle.rel_errors(_np(Y[d]), want[d])
        assert fro <= FRO_TOL and mx <= MAX_TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    # R = 16 with 16 x 8192 rows and N = 8192 needs 16 x (64 x 32 tiles) x
    # 16 B of counters (512 KiB): more than the 64 KiB static scratch.
    # Rejected from the plan alone, before any pointer is queried or
    # anything is enqueued, so this runs with or without a GPU.
    import __graft_entry__
    __graft_entry__.build()
    plan = B.fo_plan("gemm_rs", 16, 16 * 8192, 8192, 16 * 256)
    assert B.fo_workspace_size(plan) > B.FO_NOALLOC_SCRATCH_BYTES
    fake = [16 * (i + 1) for i in range(16)]
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_gemm_rs_noalloc(plan, fake, fake, fake, stream=0)
    assert e.value.code == B.FO_ERR_SCRATCH_LIMIT


@pytest.mark.gpu
def test_noalloc_call_after_a_timed_out_call_is_exact():
    # A call whose device wait runs out leaves its counters and status word in
    # the shared static array; the next call zeroes the array before it
    # launches, so a healthy call that follows gives the exact result.
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a GB300"
    dev = torch.device("cuda:0")
    R, M, K, N = 2, 256, 128, 256
    inp = gemm_rs_inputs(R, M, K, N, mode="int", seed=0)
    X = [x.to(dev) for x in inp["X"]]
    W = [w.to(dev) for w in inp["W"]]
    Y = [torch.empty(M // R, N, device=dev) for _ in range(R)]
    bad = B.fo_plan("gemm_rs", R, M, N, K * R, fault_inject="skip_signal", timeout_ns=20_000_000)
    B.fo_gemm_rs_noalloc(bad, X, W, Y)       # one counter signal is never given: the wait runs out
    torch.cuda.synchronize()
    good = B.fo_plan("gemm_rs", R, M, N, K * R)
    want = oracle.gemm_rs([_np(x) for x in inp["X"]], [_np(w) for w in inp["W"]])
    for call in range(2):
        Y = [torch.full((M // R, N), float("nan"), device=dev) for _ in range(R)]
        B.fo_gemm_rs_noalloc(good, X, W, Y)
        torch.cuda.synchronize()
        for d in range(R):
            assert np.array_equal(_np(Y[d]), want[d]), f"call {call} shard {d}"


def test_noalloc_refuses_fp32_inputs_with_w_as_k_by_n():
    # Such plans transpose W into the workspace first; the allocation-free
    # entry point has no room for that copy. Refused from the plan alone.
    import __graft_entry__
    __graft_entry__.build()
    plan = B.fo_plan("gemm_rs", 2, 64, 16, 16, in_dtype="f32")      # tiny: fits the scratch otherwise
    assert B.fo_workspace_size(plan) <= B.FO_NOALLOC_SCRATCH_BYTES
    fake = [16 * (i + 1) for i in range(2)]
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_gemm_rs_noalloc(plan, fake, fake, fake, stream=0)
    assert e.value.code == B.FO_ERR_UNSUPPORTED
