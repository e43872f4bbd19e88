"""The N > 1 host path of bench.py on CPU: world_size 2 over gloo.

Each GPU runs an independent replica (the virtual ranks of the method live on
one GPU), so the only cross-process step is the max of the per-rank timings
and the final barrier. These tests run that logic with two CPU processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, l = bench.dist_env()
        assert (w, r, l) == (world, rank, rank)
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        dist.barrier()
        out_q.put((rank, got))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(world))
    assert res == {r: 10.0 + 5.0 * (world - 1) for r in range(world)}


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_of_the_bench_workloads():
    # Operands once, output once, (R-1)/R of every fp32 partial to its owner
    # and back (reduce-scatter); peer-read all-gather moves nothing extra.
    import bench
    from ag_gemm_gb300.inputs import WORKLOADS
    rs = WORKLOADS["gemm_rs_down_r8_t8192_k1792_n4096"]
    x_w = 8 * (8192 * 1792 + 1792 * 4096) * 2
    partial = 8192 * 4096 * 4
    assert bench.algorithmic_bytes(rs) == x_w + 2 * 7 * partial + partial
    ag = WORKLOADS["ag_gemm_qkv_r4_s4096_h4096_n3072"]
    assert bench.algorithmic_bytes(ag) == (4096 * 4096 + 4 * 4096 * 3072 + 4 * 4096 * 3072) * 2
    s = bench.hbm_summary(rs, 0.5, 1.0e9, {"hbm_gbs": 6000.0})
    assert abs(s["algorithmic_gbs"] - bench.algorithmic_bytes(rs) / 0.5e-3 / 1e9) < 1e-6
    assert abs(s["traffic_gbs"] - 2000.0) < 1e-9 and abs(s["frac_algorithmic"] - s["algorithmic_gbs"] / 6000.0) < 1e-12


def test_both_arms_describe_the_workload_alike():
    # The reference arm and the GPU arm print the same `config` object.
    import bench
    from ag_gemm_gb300.inputs import WORKLOADS
    rs = WORKLOADS[bench.DEFAULT_WORKLOAD]
    c = bench.workload_config(rs, 1)
    assert c["workload"] == rs.name and (c["R"], c["M"], c["K_per_rank"], c["N"]) == (8, 8192, 1792, 4096)
    assert c["parallelism"] == "single GPU, 8 virtual ranks" and "l2" in c
    assert bench.workload_config(rs, 4)["parallelism"] == "replicas"
    ag = WORKLOADS["ag_gemm_qkv_r4_s4096_h4096_n3072"]
    assert bench.workload_config(ag, 1)["parallelism"] == "single GPU, 4 virtual ranks"


def test_oracle_sample_flop_counts_for_every_op():
    # The bench's CPU baseline counts, per pass, the FLOPs of exactly the
    # sampled output rows: R shards x rows rows x (R ranks x 2 K N) for the
    # reduce-scatters, R ranks x (R x rows) gathered rows x 2 K N_r for AG.
    import types

    import numpy as np

    import bench
    rng = np.random.default_rng(0)
    R, rows = 2, 3
    rs = types.SimpleNamespace(op="gemm_rs", R=R, dims={"M": 8, "K": 4, "N": 5})
    Xs = [rng.standard_normal((8, 4)) for _ in range(R)]
    Ws = [rng.standard_normal((4, 5)) for _ in range(R)]
    assert bench.oracle_pass(rs, (Xs, Ws), rows)[1] == 2.0 * R * rows * R * 4 * 5
    ag = types.SimpleNamespace(op="ag_gemm", R=R, dims={"M": 8, "K": 4, "N": 5})
    Xa = [rng.standard_normal((4, 4)) for _ in range(R)]
    assert bench.oracle_pass(ag, (Xa, Ws), rows)[1] == 2.0 * R * (R * rows) * 4 * 5
    dp = types.SimpleNamespace(op="dp_grad_rs", R=R, dims={"T": 6, "M": 8, "N": 5})
    Xd = [rng.standard_normal((6, 8)) for _ in range(R)]
    dY = [rng.standard_normal((6, 5)) for _ in range(R)]
    assert bench.oracle_pass(dp, (Xd, dY), rows)[1] == 2.0 * R * rows * R * 6 * 5
