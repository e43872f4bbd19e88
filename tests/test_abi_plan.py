"""CPU tests of the C ABI: the library loads, exports every declared symbol,
and fo_plan (host only) builds the schedule the oracle's reading gives."""
import os
import re

import numpy as np
import pytest

import oracle
from ag_gemm_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return B.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "flashoverlap.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fo_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTED) == names


def test_version_and_status_strings(lib):
    assert B.fo_version() == 0x000100
    for code in range(9):
        assert B.status_string(code)
    assert B.status_string(B.FO_ERR_TIMEOUT) == "device-side wait timed out"


@pytest.mark.parametrize("R", list(range(1, 17)))
def test_plan_tables_match_oracle(R):
    rs = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R)
    assert B.fo_plan_table(rs) == oracle.rs_schedule(R).tolist()
    ag = B.fo_plan("ag_gemm", R, 128 * R, 64 * R, 256)
    assert B.fo_plan_table(ag) == oracle.ag_schedule(R).tolist()
    dp = B.fo_plan("dp_grad_rs", R, 8 * R, 256, 64)
    assert B.fo_plan_table(dp) == oracle.rs_schedule(R).tolist()


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_plan_transfers_match_oracle(R):
    rs = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R)
    assert sorted(B.fo_plan_transfers(rs)) == sorted(oracle.rs_transfers(R))
    ag = B.fo_plan("ag_gemm", R, 128 * R, 64 * R, 256)
    assert sorted(B.fo_plan_transfers(ag)) == sorted(oracle.ag_transfers(R))


@pytest.mark.parametrize("R", [2, 3, 5])
def test_plan_edges_form_the_oracle_dag(R):
    rs = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R)
    got = sorted((a, b, c, d) for (a, b, c, d) in B.fo_plan_edges(rs))
    want = sorted((a[0], a[1], b[0], b[1]) for a, b in oracle.rs_dependency_edges(R))
    assert got == want


def test_sliced_schedule_is_the_ablation_table():
    R = 4
    p = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R, sched="sliced")
    assert B.fo_plan_table(p) == oracle.sliced_schedule(R).tolist()
    assert len(B.fo_plan_transfers(p)) == R * (R - 1)


def test_dropped_transfer_is_rejected():
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan("gemm_rs", 4, 512, 256, 256, fault_inject="drop_transfer")
    assert e.value.code == B.FO_ERR_PLAN_INVARIANT
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan("ag_gemm", 4, 512, 256, 256, fault_inject="drop_transfer")
    assert e.value.code == B.FO_ERR_PLAN_INVARIANT


@pytest.mark.parametrize("kw,code", [
    (dict(op="gemm_rs", R=0, M=8, N=8, K=8), B.FO_ERR_INVALID_ARG),
    (dict(op="gemm_rs", R=17, M=17, N=8, K=17), B.FO_ERR_INVALID_ARG),
    (dict(op="gemm_rs", R=3, M=8, N=8, K=24), B.FO_ERR_SHAPE),          # M % R
    (dict(op="gemm_rs", R=2, M=8, N=8, K=9), B.FO_ERR_SHAPE),           # K % R
    (dict(op="gemm_rs", R=2, M=8, N=6, K=32), B.FO_ERR_ALIGN),          # rows of W not 16 B
    (dict(op="gemm_rs", R=2, M=8, N=8, K=12), B.FO_ERR_ALIGN),          # rows of X_r not 16 B
    (dict(op="gemm_rs", R=2, M=0, N=8, K=16), B.FO_ERR_SHAPE),         # empty: no rows
    (dict(op="gemm_rs", R=2, M=8, N=0, K=16), B.FO_ERR_SHAPE),         # no columns
    (dict(op="gemm_rs", R=2, M=8, N=8, K=0), B.FO_ERR_SHAPE),          # no reduction
    (dict(op="ag_gemm", R=2, M=8, N=0, K=16), B.FO_ERR_SHAPE),
    (dict(op="ag_gemm", R=2, M=8, N=16, K=0), B.FO_ERR_SHAPE),
    (dict(op="dp_grad_rs", R=2, M=0, N=8, K=16), B.FO_ERR_SHAPE),
    (dict(op="dp_grad_rs", R=2, M=16, N=8, K=0), B.FO_ERR_SHAPE),      # no tokens
    (dict(op="gemm_a2a", R=2, M=8, N=0, K=16), B.FO_ERR_SHAPE),
    (dict(op="gemm_ar", R=2, M=8, N=8, K=0), B.FO_ERR_SHAPE),
    (dict(op="ag_gemm", R=2, M=8, N=10, K=16), B.FO_ERR_ALIGN),         # N/R = 5
    (dict(op="ag_gemm", R=3, M=9, N=8, K=16), B.FO_ERR_SHAPE),          # N % R
    (dict(op="dp_grad_rs", R=2, M=8, N=8, K=16), B.FO_ERR_ALIGN),       # M/R = 4 columns
    (dict(op="ag_gemm", R=2, M=8, N=16, K=16, out_dtype="f32"), B.FO_ERR_DTYPE),
    (dict(op="gemm_ar", R=2, M=8, N=16, K=16, out_dtype="bf16"), B.FO_ERR_DTYPE),
    (dict(op="gemm_ar", R=2, M=8, N=16, K=9), B.FO_ERR_SHAPE),
    (dict(op="gemm_rs", R=2, M=8, N=6, K=16, in_dtype="f32"), B.FO_ERR_ALIGN),   # fp32 rows of 24 bytes
    (dict(op="ag_gemm", R=2, M=8, N=16, K=16, sched="sliced"), B.FO_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_descriptors(kw, code):
    kw = dict(kw)
    op, R, M, N, K = kw.pop("op"), kw.pop("R"), kw.pop("M"), kw.pop("N"), kw.pop("K")
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan(op, R, M, N, K, **kw)
    assert e.value.code == code


def test_workspace_size_covers_counters():
    R = 8
    p = B.fo_plan("gemm_rs", R, 8192, 4096, 14336)
    tiles = (1024 // 128) * (4096 // 256)
    assert B.fo_workspace_size(p) >= 256 + R * tiles * 4 * 4
    assert B.fo_workspace_size(p) % 256 == 0


def test_launch_without_gpu_fails_loudly():
    # On a machine without a GPU (or not sm_103) a launching call must return
    # an error, never fall back to the CPU.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = B.fo_plan("gemm_rs", 2, 256, 512, 1024)
    fake = [16 * (i + 1) for i in range(2)]
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_gemm_rs(p, fake, fake, fake, 4096, stream=0)
    assert e.value.code in (B.FO_ERR_CUDA, B.FO_ERR_UNSUPPORTED)


def test_null_arguments_are_rejected():
    p = B.fo_plan("gemm_rs", 2, 256, 512, 1024)
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_gemm_rs(p, [0, 0], [16, 16], [16, 16], 4096, stream=0)
    assert e.value.code == B.FO_ERR_INVALID_ARG
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_gemm_rs(p, [24, 16], [16, 16], [16, 16], 4096, stream=0)
    assert e.value.code == B.FO_ERR_ALIGN


def test_plan_rejects_unknown_tile_config():
    d = B.PlanDesc()
    d.op, d.R, d.M, d.N, d.K = 1, 2, 256, 256, 256
    d.out_dtype = 1
    d.tile_config = 7
    import ctypes
    h = ctypes.c_void_p()
    assert B.load().fo_plan(ctypes.byref(d), ctypes.byref(h)) == B.FO_ERR_INVALID_ARG


def test_workspace_counts_pair_tiles():
    # 600-row chunks: 3 single-CTA m-tiles, 2 pair m-tiles = 4 128-row counter rows.
    p = B.fo_plan("gemm_rs", 2, 1200, 512, 512)
    assert B.fo_workspace_size(p) >= 256 + 2 * 4 * 2 * 4 * 4


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("op", ["gemm_rs", "ag_gemm", "dp_grad_rs"])
@pytest.mark.parametrize("interleave", ["auto", "lockstep", "skewed", "rank_major", "skewed_pairs"])
def test_task_order_keeps_every_ranks_schedule_order(R, op, interleave):
    dims = {"gemm_rs": (128 * R, 256, 64 * R), "ag_gemm": (128 * R, 64 * R, 256), "dp_grad_rs": (8 * R, 256, 64)}[op]
    p = B.fo_plan(op, R, *dims, interleave=interleave)
    order = B.fo_plan_task_order(p)
    assert sorted(order) == [(r, s) for r in range(R) for s in range(R)]
    for r in range(R):
        steps = [s for (rr, s) in order if rr == r]
        assert steps == list(range(R))            # each rank runs its own steps in order


@pytest.mark.parametrize("R", [2, 3, 4, 8])
def test_skewed_order_groups_partials_by_owner_in_step_order(R):
    p = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R, interleave="skewed")
    order = B.fo_plan_task_order(p)
    table = oracle.rs_schedule(R)
    chunks = [int(table[r, s]) for (r, s) in order]
    # runs of equal owners: slots t = s - r; every slot sends to one owner
    slots = {}
    for (r, s), c in zip(order, chunks):
        slots.setdefault(s - r, set()).add(c)
    assert all(len(v) == 1 for v in slots.values())
    # every owner gets its partials in step order (first partial stored first)
    for c in range(R):
        steps = [s for (r, s), cc in zip(order, chunks) if cc == c]
        assert steps == sorted(steps) == list(range(R))


@pytest.mark.parametrize("R", [2, 3, 4, 5, 8, 16])
def test_skewed_pairs_run_each_ranks_two_steps_of_a_slot_pair_together(R):
    p = B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R, interleave="skewed_pairs")
    order = B.fo_plan_task_order(p)
    assert sorted(order) == [(r, s) for r in range(R) for s in range(R)]
    table = oracle.rs_schedule(R)
    # slots t = s - r, taken in pairs (-(R-1), -(R-2)), (-(R-3), -(R-4)), ...
    pair_of = lambda r, s: (s - r + R - 1) // 2
    pairs = [pair_of(r, s) for (r, s) in order]
    assert pairs == sorted(pairs)
    for k in set(pairs):
        tasks = [(r, s) for (r, s) in order if pair_of(r, s) == k]
        # at most two owners per slot pair, and a rank's tasks of the pair adjacent and in step order
        assert len({int(table[r, s]) for (r, s) in tasks}) <= 2
        for r in {r for (r, _) in tasks}:
            idx = [i for i, (rr, _) in enumerate(tasks) if rr == r]
            assert idx == list(range(idx[0], idx[0] + len(idx)))
            assert [tasks[i][1] for i in idx] == sorted(tasks[i][1] for i in idx)
    # every owner still gets its partials in step order
    for c in range(R):
        steps = [s for (r, s) in order if int(table[r, s]) == c]
        assert steps == list(range(R))


def test_auto_interleave_per_op_and_transport():
    R = 4
    rs = B.fo_plan_task_order(B.fo_plan("gemm_rs", R, 512, 256, 256))
    assert rs == B.fo_plan_task_order(B.fo_plan("gemm_rs", R, 512, 256, 256, interleave="skewed_pairs"))
    ar = B.fo_plan_task_order(B.fo_plan("gemm_ar", R, 512, 256, 256))
    assert ar == rs
    ag = B.fo_plan_task_order(B.fo_plan("ag_gemm", R, 512, 256, 256))
    assert ag == [(r, s) for r in range(R) for s in range(R)]
    dp = B.fo_plan_task_order(B.fo_plan("dp_grad_rs", R, 512, 256, 256))
    assert dp == [(r, s) for r in range(R) for s in range(R)]
    lock = B.fo_plan_task_order(B.fo_plan("ag_gemm", R, 512, 256, 256, interleave="lockstep"))
    assert lock == [(r, s) for s in range(R) for r in range(R)]
    # the ring reduce-scatter runs lockstep: a chain's hops a whole step apart
    for op in ("gemm_rs", "dp_grad_rs"):
        ring = B.fo_plan_task_order(B.fo_plan(op, R, 512, 256, 256, rs_algo="ring"))
        assert ring == B.fo_plan_task_order(B.fo_plan(op, R, 512, 256, 256, rs_algo="ring", interleave="lockstep"))
    # so does the ring-forwarded all-gather (copy transport)
    copy = B.fo_plan_task_order(B.fo_plan("ag_gemm", R, 512, 256, 256, ag_transport="copy"))
    assert copy == lock


def test_copy_transport_requires_gather_buffers():
    p = B.fo_plan("ag_gemm", 2, 256, 256, 256, ag_transport="copy")
    fake = [16 * (i + 1) for i in range(2)]
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_ag_gemm(p, fake, fake, fake, None, 4096, stream=0)
    assert e.value.code == B.FO_ERR_INVALID_ARG


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_allreduce_plan_is_rs_then_allgather(R):
    p = B.fo_plan("gemm_ar", R, 128 * R, 256, 64 * R)
    assert B.fo_plan_table(p) == oracle.rs_schedule(R).tolist()
    assert sorted(B.fo_plan_transfers(p)) == sorted(oracle.ar_transfers(R))


def test_bf16_output_keeps_fp32_sums_in_the_workspace():
    R, M, N, K = 8, 8192, 4096, 14336
    f32 = B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K))
    b16 = B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K, out_dtype="bf16"))
    assert b16 - f32 >= M * N * 4
    with pytest.raises(B.FlashOverlapError) as e:     # the allocation-free entry point keeps fp32 only
        B.fo_gemm_rs_noalloc(B.fo_plan("gemm_rs", 2, 256, 256, 256, out_dtype="bf16"), [16, 32], [16, 32],
                             [16, 32], stream=0)
    assert e.value.code in (B.FO_ERR_SCRATCH_LIMIT, B.FO_ERR_DTYPE)


# ------------------------------------------------------------------ ring reduce-scatter

def _ring_plan(op, R, **kw):
    if op == "gemm_rs":
        return B.fo_plan("gemm_rs", R, 128 * R, 256, 64 * R, rs_algo="ring", **kw)
    return B.fo_plan("dp_grad_rs", R, 8 * R, 256, 64, rs_algo="ring", **kw)


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("op", ["gemm_rs", "dp_grad_rs"])
def test_ring_plan_transfers_match_oracle(R, op):
    p = _ring_plan(op, R)
    assert B.fo_plan_table(p) == oracle.rs_schedule(R).tolist()
    assert sorted(B.fo_plan_transfers(p)) == sorted(oracle.rs_transfers(R, ring=True))


@pytest.mark.parametrize("R", [2, 3, 5, 8])
def test_ring_plan_edges_are_program_order_and_forwards(R):
    p = _ring_plan("gemm_rs", R)
    table = B.fo_plan_table(p)
    want = [(r, s, r, s + 1) for r in range(R) for s in range(R - 1)]
    want += [(r, s, (r + 1) % R, s + 1) for s in range(R - 1) for r in range(R)]
    assert sorted(B.fo_plan_edges(p)) == sorted(want)
    # every forward reaches the rank that handles the same chunk next
    for (src, dst, c, s) in B.fo_plan_transfers(p):
        assert table[src][s] == c and table[dst][s + 1] == c


@pytest.mark.parametrize("R", [2, 3, 4, 8, 16])
@pytest.mark.parametrize("op", ["gemm_rs", "dp_grad_rs"])
@pytest.mark.parametrize("interleave", ["auto", "lockstep", "skewed", "skewed_pairs"])
def test_ring_kernel_order_runs_every_chain_in_hop_order(R, op, interleave):
    # The kernel adds a chunk's partials in the order it runs them, and a
    # hop waits for its predecessor: each chain must run in hop order, or a
    # wait could target a task that has not started.
    p = _ring_plan(op, R, interleave=interleave)
    table = B.fo_plan_table(p)
    pos = {rs: i for i, rs in enumerate(B.fo_plan_task_order(p))}
    for c in range(R):
        chain = [((c + 1 + s) % R, s) for s in range(R)]
        assert all(table[r][s] == c for r, s in chain)
        assert [pos[t] for t in chain] == sorted(pos[t] for t in chain)


@pytest.mark.parametrize("op,kw,code", [
    ("gemm_rs", dict(interleave="rank_major"), B.FO_ERR_UNSUPPORTED),   # chains out of hop order
    ("dp_grad_rs", dict(interleave="rank_major"), B.FO_ERR_UNSUPPORTED),
    ("gemm_rs", dict(sched="sliced"), B.FO_ERR_UNSUPPORTED),             # no chunk passes along the ring
    ("gemm_ar", {}, B.FO_ERR_UNSUPPORTED),
    ("ag_gemm", {}, B.FO_ERR_INVALID_ARG),
    ("gemm_rs", dict(fault_inject="drop_transfer"), B.FO_ERR_PLAN_INVARIANT),
])
def test_ring_plan_rejections(op, kw, code):
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan(op, 4, 512, 256, 256, rs_algo="ring", **kw)
    assert e.value.code == code


def test_ring_workspace_holds_every_ranks_receive_buffer():
    R, M, N, K = 8, 8192, 4096, 14336
    direct = B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K))
    ring = B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K, rs_algo="ring"))
    assert ring - direct >= R * M * N * 4
    # a bf16 ring output needs no separate fp32 shard sums
    assert B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K, rs_algo="ring", out_dtype="bf16")) == ring
    with pytest.raises(B.FlashOverlapError) as e:     # the allocation-free entry point is direct-only
        B.fo_gemm_rs_noalloc(B.fo_plan("gemm_rs", 2, 256, 256, 256, rs_algo="ring"), [16, 32], [16, 32],
                             [16, 32], stream=0)
    assert e.value.code == B.FO_ERR_UNSUPPORTED


# ------------------------------------------------------------------ tracing, delay injection, logging

def test_trace_plan_reserves_timestamps_in_the_workspace():
    R, M, N, K = 8, 8192, 4096, 14336
    plain = B.fo_workspace_size(B.fo_plan("gemm_rs", R, M, N, K))
    traced = B.fo_plan("gemm_rs", R, M, N, K, trace=True)
    assert B.fo_workspace_size(traced) - plain >= B.FO_TRACE_MAX_CTAS * B.FO_TRACE_STAMPS * 8
    with pytest.raises(B.FlashOverlapError) as e:        # nothing launched yet
        B.fo_trace_query(traced, 4096)
    assert e.value.code == B.FO_ERR_INVALID_ARG
    with pytest.raises(B.FlashOverlapError) as e:        # plan built without trace
        B.fo_trace_query(B.fo_plan("gemm_rs", R, M, N, K), 4096)
    assert e.value.code == B.FO_ERR_INVALID_ARG
    with pytest.raises(B.FlashOverlapError) as e:        # the timestamps alone fill the static scratch
        B.fo_gemm_rs_noalloc(B.fo_plan("gemm_rs", 2, 256, 256, 256, trace=True), [16, 32], [16, 32], [16, 32],
                             stream=0)
    assert e.value.code == B.FO_ERR_SCRATCH_LIMIT


@pytest.mark.parametrize("kw", [
    dict(inject_delay_us=100),                                         # a delay without its hook
    dict(fault_inject="delay_first_task", inject_delay_us=-1),
    dict(fault_inject="delay_first_task", inject_delay_us=1_000_001),
])
def test_delay_injection_arguments_are_checked(kw):
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan("gemm_rs", 4, 512, 256, 256, **kw)
    assert e.value.code == B.FO_ERR_INVALID_ARG


def test_trace_summary_reads_the_tail_off_the_stamps():
    rows = [[100, 900, 950, 990, 940, 960, 1000, 0],   # leader: MMAs done at 900, last transfer 990
            [105, 0, 930, 935, 1020, 925, 1030, 0]]    # peer: its epilogue finishes last
    s = B.trace_summary(rows)
    assert s == {"span_ns": 930, "mma_end_ns": 800, "transfers_end_ns": 920, "exposed_tail_ns": 120}


def test_fo_log_prints_plans_to_stderr():
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, '.'); from ag_gemm_gb300 import binding as B; "
            "B.fo_plan('gemm_rs', 4, 1024, 512, 256, rs_algo='ring')")
    env = dict(os.environ, FO_LOG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "[flashoverlap] plan gemm_rs R=4 M=1024 N=512 K=256" in r.stderr and "ring RS" in r.stderr
    env["FO_LOG"] = "0"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert "[flashoverlap]" not in r.stderr


def test_binding_refuses_host_tensors():
    # A CPU tensor never reaches the library: its address would not be
    # device memory.
    import torch
    p = B.fo_plan("gemm_rs", 2, 256, 256, 512)
    host = [torch.zeros(256, 256, dtype=torch.bfloat16) for _ in range(2)]
    with pytest.raises(ValueError):
        B.fo_gemm_rs(p, host, host, host, 4096, stream=0)
    assert B.fo_plan_last_launches(p) == 0
    assert B.fo_check_device_pointers.__doc__


# ------------------------------------------------------------------ all-to-all (Ulysses projection)

@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
def test_a2a_plan_matches_the_oracle(R):
    p = B.fo_plan("gemm_a2a", R, 128 * R, 64 * R, 256)
    assert B.fo_plan_table(p) == oracle.rs_schedule(R).tolist()          # the block that stays comes last
    assert sorted(B.fo_plan_transfers(p)) == sorted(oracle.a2a_transfers(R))
    got = sorted((a, b, c, d) for (a, b, c, d) in B.fo_plan_edges(p))
    want = sorted((a[0], a[1], b[0], b[1]) for a, b in oracle.rs_dependency_edges(R))
    assert got == want
    assert B.fo_plan_task_order(p) == [(r, s) for r in range(R) for s in range(R)]   # AUTO: rank-major


def test_a2a_plan_options_and_workspace():
    R = 8
    p = B.fo_plan("gemm_a2a", R, 8192, 12288, 4096)
    sl = B.fo_plan("gemm_a2a", R, 8192, 12288, 4096, sched="sliced")
    assert B.fo_plan_table(sl) == oracle.sliced_schedule(R).tolist()
    # no readiness counters: the header, plus the tail split's buffers when the
    # launch's last wave would idle most units
    small = B.fo_plan("gemm_a2a", 2, 512, 512, 256, tail_split="off")
    assert B.fo_workspace_size(small) == 256
    assert B.fo_workspace_size(p) > 256


@pytest.mark.parametrize("kw,code", [
    (dict(R=2, M=8, N=15, K=16), B.FO_ERR_SHAPE),                        # N not divisible by R
    (dict(R=2, M=8, N=12, K=16), B.FO_ERR_ALIGN),                        # N/R = 6 columns: not 16 bytes
    (dict(R=2, M=8, N=16, K=12), B.FO_ERR_ALIGN),                        # rows of X_r not 16 bytes
    (dict(R=2, M=8, N=16, K=16, out_dtype="f32"), B.FO_ERR_DTYPE),
    (dict(R=2, M=8, N=16, K=16, in_dtype="f32"), B.FO_ERR_DTYPE),
    (dict(R=2, M=8, N=16, K=16, rs_algo="ring"), B.FO_ERR_INVALID_ARG),
    (dict(R=2, M=8, N=16, K=16, ag_transport="copy"), B.FO_ERR_INVALID_ARG),
    (dict(R=2, M=9, N=16, K=16), B.FO_ERR_SHAPE),
])
def test_a2a_plan_rejections(kw, code):
    kw = dict(kw)
    R, M, N, K = kw.pop("R"), kw.pop("M"), kw.pop("N"), kw.pop("K")
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_plan("gemm_a2a", R, M, N, K, **kw)
    assert e.value.code == code


def test_a2a_plan_refuses_the_reduce_scatter_calls():
    p = B.fo_plan("gemm_a2a", 2, 256, 512, 256)
    fake = [16 * (i + 1) for i in range(2)]
    for call in (lambda: B.fo_gemm_rs(p, fake, fake, fake, 4096, stream=0),
                 lambda: B.fo_gemm_partials(p, fake, fake, fake, 4096, stream=0),
                 lambda: B.fo_reduce_scatter_f32(p, fake, fake, stream=0),
                 lambda: B.fo_all_gather_copy(p, fake, fake, stream=0)):
        with pytest.raises(B.FlashOverlapError) as e:
            call()
        assert e.value.code == B.FO_ERR_INVALID_ARG
    rs = B.fo_plan("gemm_rs", 2, 256, 512, 256)
    for call in (lambda: B.fo_gemm_a2a(rs, fake, fake, fake, 4096, stream=0),
                 lambda: B.fo_all_to_all_copy(rs, fake, fake, stream=0)):
        with pytest.raises(B.FlashOverlapError) as e:
            call()
        assert e.value.code == B.FO_ERR_INVALID_ARG


def test_fp32_inputs_take_either_weight_layout():
    # The 256 x 512 x 512 R = 2 integer workload as stated: fp32 X_r [256 x 512]
    # and W_r [512 x 512] in the [K x N] layout (tf32 MMA, B operand MN-major).
    for layout in ("kn", "nk"):
        p = B.fo_plan("gemm_rs", 2, 256, 512, 1024, in_dtype="f32", w_layout=layout)
        assert B.fo_plan_table(p) == oracle.rs_schedule(2).tolist()


# ------------------------------------------------------------------ query-split attention: host checks

def test_attn_rs_rejects_bad_arguments_on_the_host():
    fake = [16 * (i + 1) for i in range(2)]
    p = B.fo_plan("gemm_rs", 2, 512, 256, 2 * 2 * 128)          # T = 512, heads = 2 per rank, H = 256
    for heads, causal, code in ((0, 0, B.FO_ERR_INVALID_ARG), (2, 2, B.FO_ERR_INVALID_ARG),
                                (3, 0, B.FO_ERR_SHAPE)):         # K != R * heads * 128
        with pytest.raises(B.FlashOverlapError) as e:
            B._check(B.load().fo_attn_rs(p, B._ptr_array(fake), B._ptr_array(fake), B._ptr_array(fake),
                                         B._ptr_array(fake), B._ptr_array(fake), B._ptr_array(fake), heads, causal,
                                         4096, 0), "fo_attn_rs")
        assert e.value.code == code
    odd = B.fo_plan("gemm_rs", 2, 384, 256, 2 * 128)              # T/R = 192: not whole 128-row tiles
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_attn_rs(odd, fake, fake, fake, fake, fake, fake, 1, False, 4096, stream=0)
    assert e.value.code == B.FO_ERR_SHAPE
    ag = B.fo_plan("ag_gemm", 2, 512, 256, 256)
    with pytest.raises(B.FlashOverlapError) as e:
        B.fo_attn_rs(ag, fake, fake, fake, fake, fake, fake, 1, False, 4096, stream=0)
    assert e.value.code == B.FO_ERR_INVALID_ARG


def test_attention_alone_rejects_bad_arguments_on_the_host():
    fake = [16 * (i + 1) for i in range(2)]

    def call(plan, heads, causal, V=fake):
        B._check(B.load().fo_attention(plan, B._ptr_array(fake), B._ptr_array(fake), B._ptr_array(V),
                                       B._ptr_array(fake), heads, causal, 4096, 0), "fo_attention")

    p = B.fo_plan("gemm_rs", 2, 512, 256, 2 * 2 * 128)
    f32 = B.fo_plan("gemm_rs", 2, 512, 256, 2 * 2 * 128, in_dtype="f32")
    for plan, heads, causal, V, code in ((p, 0, 0, fake, B.FO_ERR_INVALID_ARG),
                                         (p, 2, 2, fake, B.FO_ERR_INVALID_ARG),
                                         (p, 3, 0, fake, B.FO_ERR_SHAPE),          # K != R * heads * 128
                                         (p, 2, 1, [16, 0], B.FO_ERR_INVALID_ARG),  # a null V pointer
                                         (p, 2, 1, [16, 24], B.FO_ERR_ALIGN),       # V not 16-byte aligned
                                         (f32, 2, 1, fake, B.FO_ERR_INVALID_ARG)):  # fp32 inputs
        with pytest.raises(B.FlashOverlapError) as e:
            call(plan, heads, causal, V)
        assert e.value.code == code


def test_partials_sharded_rejects_bad_arguments_on_the_host():
    fake = [16 * (i + 1) for i in range(4)]
    dp = B.fo_plan("dp_grad_rs", 4, 512, 256, 1024)
    for plan, A, code in ((B.fo_plan("gemm_rs", 4, 512, 256, 1024), fake, B.FO_ERR_INVALID_ARG),
                          (B.fo_plan("ag_gemm", 4, 512, 256, 1024), fake, B.FO_ERR_INVALID_ARG),
                          (B.fo_plan("dp_grad_rs", 4, 512, 256, 1026), fake, B.FO_ERR_SHAPE),  # T % R
                          (B.fo_plan("dp_grad_rs", 4, 512, 256, 1040), fake, B.FO_ERR_SHAPE),  # T/R % 64
                          (dp, [16, 32, 0, 64], B.FO_ERR_INVALID_ARG),              # a null shard
                          (dp, [16, 32, 40, 64], B.FO_ERR_ALIGN)):                  # a shard off 16 bytes
        with pytest.raises(B.FlashOverlapError) as e:
            B.fo_gemm_partials_sharded(plan, A, fake, fake, 4096, stream=0)
        assert e.value.code == code
