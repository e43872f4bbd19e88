#!/usr/bin/env python
"""Benchmark of the fused GEMM + reduce-scatter (FlashOverlap Flash-RS) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras]

One step = one fo_gemm_rs call over the whole workload: R = 8 virtual ranks,
each X_r [8192 x 1792] . W_r [1792 x 4096] (bf16, fp32 accumulate), the
partials reduce-scattered by rows into eight [1024 x 4096] fp32 shards (the
TP-SP MLP down-projection: 8192 tokens, FFN 14336 / 8 per rank, hidden 4096).
Inputs are seeded synthetic tensors (X ~ N(0,1), W ~ N(0,0.02)) already
resident in HBM; together they exceed L2, so no L2 flush runs between steps.

The JSON line reports whole-job TFLOP/s, the roofline fraction of the fused
kernel against the measured bf16 dense peak, short timed loops of the other
fused ops (all-gather QKV projection, DP gradient, all-to-all projection,
query-split attention with its projection, the TP-SP layer's forward and
backward) on the same device, the same metric end to end with
host buffers (host->device inputs and device->host outputs inside the timed
region), the CPU oracle timed on a bounded sample, and, next to them, the
pure-GEMM control, the unfused baseline (our GEMM + a separate reduce kernel),
the data-slicing baseline over chunk counts 1 to 16, and cuBLAS through
torch.matmul.

With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica on its own GPU (the method here needs no cross-GPU exchange: the R
ranks are buffers on one GPU); value = all ranks' FLOPs / max time.

--impl reference times the CPU oracle (fp64 numpy) on a bounded sample of
the same workload, rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+RS/AG TFLOP/s (R virtual ranks, 1 GB300), % of bf16 tensor peak"
DEFAULT_WORKLOAD = "gemm_rs_down_r8_t8192_k1792_n4096"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic_bytes(w) -> float:
    """DRAM bytes a launch must move at least: operands read once, the
    output written once, and for a reduce-scatter (R-1)/R of every rank's
    fp32 partial written to its owner and read back; peer-read all-gather
    moves no extra bytes."""
    d, R = w.dims, w.R
    if w.op == "gemm_rs":
        M, K, N = d["M"], d["K"], d["N"]
        eb = 4 if w.dtype == "f32" else 2
        return R * (M * K + K * N) * eb + 2.0 * (R - 1) * M * N * 4 + M * N * 4
    if w.op == "gemm_ar":
        # The reduce-scatter's bytes, with the fp32 result written into all
        # R ranks' full outputs instead of once.
        M, K, N = d["M"], d["K"], d["N"]
        return R * (M * K + K * N) * 2 + 2.0 * (R - 1) * M * N * 4 + R * M * N * 4
    if w.op == "dp_grad_rs":
        T, M, N = d["T"], d["M"], d["N"]
        return R * (T * M + T * N) * 2 + 2.0 * (R - 1) * M * N * 4 + M * N * 4
    if w.op == "ag_gemm":
        M, K, N = d["M"], d["K"], d["N"]
        return (M * K + R * K * N + R * M * N) * 2
    if w.op == "gemm_a2a":
        # X once, every rank's whole W_r once, Y once; the all-to-all's
        # transfer is the output store itself.
        M, K, N = d["M"], d["K"], d["N"]
        return (M * K + R * K * N + M * N) * 2
    raise ValueError(w.op)


def hbm_summary(w, kernel_ms, traffic, peaks):
    """Bytes per launch and GB/s against the measured copy bandwidth."""
    alg = algorithmic_bytes(w)
    peak = float(peaks["hbm_gbs"])
    out = {"algorithmic_bytes": alg, "algorithmic_gbs": alg / (kernel_ms * 1e-3) / 1e9, "peak_gbs": peak,
           "traffic_bytes": traffic, "traffic_gbs": None}
    out["frac_algorithmic"] = out["algorithmic_gbs"] / peak
    if traffic:
        out["traffic_gbs"] = traffic / (kernel_ms * 1e-3) / 1e9
    return out


GEMM_SOURCES = ("fo_device.cuh", "fo_kernel.cuh", "fo_plan.cpp")
ATTN_SOURCES = ("fo_device.cuh", "fo_attn.cu")


def kernel_source_sha256(sources=GEMM_SOURCES) -> str:
    """sha256 of the kernel and plan sources with comments and blank lines
    removed, so that a profile stays tied to the code it measured and not to
    its comments."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "ag_gemm_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
        h.update(src.encode("utf-8"))
    return h.hexdigest()


def profiled_traffic(workload_name: str, sources=GEMM_SOURCES, prefix="fused"):
    """DRAM bytes per launch of the workload's dominant kernel from its
    committed ncu summary, or None when that capture was taken on other
    kernel source than the one built now."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload_name}.md")
    if not os.path.exists(path):
        return None
    sha = traffic = None
    with open(path) as f:
        for line in f:
            if line.startswith("kernel_source_sha256:"):
                sha = line.split(":", 1)[1].strip()
            elif line.startswith("traffic_bytes_per_launch:"):
                traffic = float(line.split(":", 1)[1].strip())
    if sha and traffic and sha == kernel_source_sha256(sources):
        return traffic
    return None


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"fo_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def mark(self, what: str):
        setattr(self, what, time.time())

    def summary(self):
        """Median SM clock and throttle reasons over the samples taken between
        mark("t0") and mark("t1") (all samples if fewer than 3 fall inside)."""
        if self.proc is None or not os.path.exists(self.path):
            return None
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    sm = float(parts[1])
                    mx = float(parts[2])
                except ValueError:
                    continue
                samples.append((ts, sm, mx, [n for n, v in zip(names, parts[5:9]) if v.lower().startswith("active")]))
        if not samples:
            return None
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        inside = [x for x in samples if t0 is not None and t1 is not None and t0 - 0.05 <= x[0] <= t1 + 0.05]
        used = inside if len(inside) >= 3 else samples
        sms = sorted(x[1] for x in used)
        reasons = sorted({r for x in used for r in x[3]})
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": max(x[2] for x in used), "reasons": reasons,
                "samples": len(used), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------- CPU oracle timing

def oracle_inputs(workload):
    """The workload's seeded inputs as the float64 arrays the oracle takes:
    (X, W) for GEMM-RS and AG-GEMM, (X, dY) for DP-grad-RS."""
    inp = workload.make()
    second = inp["dY"] if workload.op == "dp_grad_rs" else inp["W"]
    return [x.double().numpy() for x in inp["X"]], [w.double().numpy() for w in second]


def oracle_pass(workload, arrays, rows: int):
    """One pass of the CPU oracle over the first `rows` rows of every output
    shard (of every source shard of every rank's output, for AG-GEMM);
    returns (seconds, FLOPs)."""
    import numpy as np

    import oracle
    d, R = workload.dims, workload.R
    A, Bn = arrays
    idx = np.arange(rows)
    t0 = time.perf_counter()
    if workload.op in ("gemm_rs", "gemm_ar"):
        # (The all-reduce's rows of shard sh are the reduce-scatter's, the
        # same in every rank's output.)
        for sh in range(R):
            oracle.gemm_rs_rows(A, Bn, sh, idx)
        flops = 2.0 * R * rows * R * d["K"] * d["N"]
    elif workload.op == "ag_gemm":
        rpc = d["M"] // R
        g = np.concatenate([src * rpc + idx for src in range(R)])
        for r in range(R):
            oracle.ag_gemm_rows(A, Bn, r, g)
        flops = 2.0 * R * len(g) * d["K"] * d["N"]
    elif workload.op == "gemm_a2a":
        rpc = d["M"] // R
        g = np.concatenate([src * rpc + idx for src in range(R)])
        for c in range(R):
            oracle.gemm_a2a_rows(A, Bn, c, g)
        flops = 2.0 * R * len(g) * d["K"] * (d["N"] // R)
    else:
        for sh in range(R):
            oracle.dp_grad_rs_rows(A, Bn, sh, idx)
        flops = 2.0 * R * rows * R * d["T"] * d["N"]
    return time.perf_counter() - t0, flops


def oracle_rows_for(workload, arrays, target_s: float) -> int:
    """Rows per shard whose oracle pass takes about target_s (doubling from 4,
    at most the whole shard)."""
    rpc = workload.dims["M"] // workload.R
    rows = 4
    while rows < rpc:
        dt, _ = oracle_pass(workload, arrays, rows)
        if dt >= target_s / 2:
            break
        rows = min(rpc, rows * 2)
    return rows


def oracle_sample(workload, arrays, budget_s: float = 12.0):
    """Time the oracle for about budget_s on a bounded sample of the workload:
    (TFLOP/s, description)."""
    rows = oracle_rows_for(workload, arrays, min(budget_s, 4.0))
    tot_t = tot_f = 0.0
    passes = 0
    while tot_t < budget_s and passes < 10:
        dt, fl = oracle_pass(workload, arrays, rows)
        tot_t += dt
        tot_f += fl
        passes += 1
    what = {"ag_gemm": "source shards of every rank's output",
            "gemm_a2a": "source ranks' row blocks of every rank's output"}.get(workload.op, "output shards")
    desc = (f"{passes} pass(es) over {rows} of {workload.dims['M'] // workload.R} rows of each of the "
            f"{workload.R} {what} ({tot_f / 1e9:.0f} GFLOP fp64, {tot_t:.1f} s)")
    return tot_f / tot_t / 1e12, desc


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def workload_config(w, world: int) -> dict:
    """The `config` object of a bench line, the same for both arms."""
    dims = dict(w.dims)
    if w.op in ("gemm_rs", "gemm_ar"):
        dims = {"M": dims["M"], "K_per_rank": dims["K"], "N": dims["N"]}
        out_mb = (w.R if w.op == "gemm_ar" else 1) * dims["M"] * dims["N"] * 4 / 1e6
        in_mb = w.R * (dims["M"] * dims["K_per_rank"] + dims["K_per_rank"] * dims["N"]) * \
            (4 if w.dtype == "f32" else 2) / 1e6
        if in_mb + out_mb > 129:
            l2 = f"no flush: inputs ({in_mb:.0f} MB) and output ({out_mb:.0f} MB) of a step exceed the 129 MB L2"
        else:
            l2 = f"inputs ({in_mb:.1f} MB) and output ({out_mb:.1f} MB) fit in the 129 MB L2: a parity case"
    else:
        l2 = "no flush: a step's operands exceed the 129 MB L2"
    return {"workload": w.name, "R": w.R, **dims, "l2": l2,
            "parallelism": "replicas" if world > 1 else f"single GPU, {w.R} virtual ranks"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from ag_gemm_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    arrays = oracle_inputs(w)
    rows = oracle_rows_for(w, arrays, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    per = []
    for i in range(args.warmup + args.steps):
        dt, fl = oracle_pass(w, arrays, rows)
        if i >= args.warmup:
            per.append((dt, fl))
    tot_t = sum(p[0] for p in per)
    tot_flops = sum(p[1] for p in per)
    value = tot_flops / tot_t / 1e12
    what = {"ag_gemm": "source shards of every rank's output",
            "gemm_a2a": "source ranks' row blocks of every rank's output"}.get(w.op, "output shards")
    desc = (f"per step: {rows} of {w.dims['M'] // w.R} rows of each of the {w.R} {what} "
            f"({per[0][1] / 1e9:.0f} GFLOP fp64 numpy)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(per),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def measure_e2e(B, mk_plan, launch, host_in, dev_in, dev_out, dev, stream, world, flops, steps):
    """The metric end to end through the public API with host buffers. Every
    step copies its inputs (each tensor of host_in) in from pinned host
    memory and its outputs out to pinned host memory. Steps are pipelined
    over two device buffer sets: step j+1's inputs stream in and step j-1's
    outputs stream out (copy engines, two more streams) while step j
    computes. dev_in / dev_out are the first buffer set; mk_plan() makes a
    plan per set (each keeps its parameter block cached); launch(plan, ins,
    outs, ws, stream) is the call."""
    import torch
    import torch.distributed as dist
    hin = [[t.pin_memory() for t in group] for group in host_in]
    hout = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in dev_out] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for group in hin for t in group)
    d2h = sum(t.numel() * t.element_size() for t in hout[0])
    sets = [(dev_in, dev_out),
            ([[torch.empty_like(t) for t in group] for group in dev_in], [torch.empty_like(o) for o in dev_out])]
    plans = [mk_plan(), mk_plan()]
    wss = []
    for p in plans:
        ws = torch.empty(B.fo_workspace_size(p), dtype=torch.uint8, device=dev)
        B.fo_workspace_init(p, ws, stream)
        wss.append(ws)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def run(nsteps):
        in_ready = [torch.cuda.Event() for _ in range(nsteps)]
        done = [torch.cuda.Event() for _ in range(nsteps)]
        out_done = [torch.cuda.Event() for _ in range(nsteps)]
        for j in range(nsteps):
            din, dout = sets[j % 2]
            with torch.cuda.stream(s_in):
                if j >= 2:
                    s_in.wait_event(done[j - 2])          # set j%2's inputs no longer read
                for dgroup, hgroup in zip(din, hin):
                    for d_, h_ in zip(dgroup, hgroup):
                        d_.copy_(h_, non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            if j >= 2:
                stream.wait_event(out_done[j - 2])        # set j%2's outputs already copied out
            launch(plans[j % 2], din, dout, wss[j % 2], stream)
            done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[j])
                for h_, d_ in zip(hout[j % 2], dout):
                    h_.copy_(d_, non_blocking=True)
                out_done[j].record(s_out)
        stream.wait_event(out_done[nsteps - 1])

    run(2)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev) / steps
    for p, ws in zip(plans, wss):
        code, info = B.fo_status_query(p, ws, stream)
        if code != 0:
            raise RuntimeError(f"device status {code} {info}")
    return {"value": world * flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": "inputs of step j+1 in and outputs of step j-1 out during step j"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    from ag_gemm_gb300 import binding as B
    from ag_gemm_gb300.inputs import WORKLOADS

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    if args.workload == LAYER_WORKLOAD:
        return run_layer(args, dev, world, rank)
    if args.workload == ATTN_WORKLOAD:
        return run_attn(args, dev, world, rank)
    w = WORKLOADS[args.workload]
    if w.op != "gemm_rs":
        return run_other_op(args, w, dev, world, rank)
    R, M, K, N = w.R, w.dims["M"], w.dims["K"], w.dims["N"]
    flops = w.flops()
    peaks, peak_src = load_peaks()

    inp = w.make()
    X = [x.to(dev) for x in inp["X"]]
    W = [x.to(dev) for x in inp["W"]]
    Y = [torch.empty(M // R, N, dtype=torch.float32, device=dev) for _ in range(R)]
    plan = B.fo_plan("gemm_rs", R, M, N, K * R)
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)
    stream = torch.cuda.current_stream(dev)

    def step():
        B.fo_gemm_rs(plan, X, W, Y, ws, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    code, info = B.fo_status_query(plan, ws, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} {info}")

    # The timed region holds nothing but the fused kernel's launches, back
    # to back on one stream: its average launch duration is the region's
    # CUDA-event time over the launch count (events between the launches
    # would add their own gaps).
    launches = 0
    with ClockSampler(_smi_id(dev)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        clk.mark("t0")
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step()
            launches += B.fo_plan_last_launches(plan)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("t1")
        if world > 1:
            dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    code, info = B.fo_status_query(plan, ws, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} {info}")
    kernel_ms = elapsed_ms / args.steps   # one launch a step
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    ms_per_step = elapsed_ms / args.steps
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    # A timed region of a quarter second or more of back-to-back launches
    # runs under the power cap: compare with the sustained measured peak;
    # shorter bursts with the burst peak.
    sustained = elapsed_ms >= 250.0
    peak = float(peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
    peak_name = "bf16_tflops_sustained" if sustained else "bf16_tflops (burst)"

    e2e = measure_e2e(B, lambda: B.fo_plan("gemm_rs", R, M, N, K * R),
                      lambda p, din, dout, ws_, s_: B.fo_gemm_rs(p, din[0], din[1], dout, ws_, s_),
                      [inp["X"], inp["W"]], [X, W], Y, dev, stream, world, flops, max(4, min(args.steps, 12)))

    extras = {}
    others = None
    if not args.no_extras:
        extras = measure_extras(B, plan, X, W, Y, ws, stream, flops, dev)
        others = measure_other_workloads(B, dev, stream)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": args.traffic if args.traffic is not None else profiled_traffic(w.name),
                     "peak_source": f"{peak_name}, {peak_src}",
                     "frac_of_burst_peak": achieved / float(peaks["bf16_tflops"])},
        "hbm": hbm_summary(w, kernel_ms, args.traffic if args.traffic is not None else profiled_traffic(w.name),
                           peaks),
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "baselines": extras,
        "other_workloads": others,
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, desc = oracle_sample(w, oracle_inputs(w))
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


LAYER_WORKLOAD = "tpsp_layer_r8_t8192_h4096_f14336"


def _op_setup(B, w, dev):
    """Device inputs, outputs, plan and workspace of an AG-GEMM, A2A, AR or
    DP-grad-RS workload: (inp, A, Bm, Y, plan, ws, launch(stream))."""
    import torch
    d = w.dims
    inp = w.make()
    if w.op == "gemm_a2a":
        R, M, K, N = w.R, d["M"], d["K"], d["N"]
        A = [x.to(dev) for x in inp["X"]]
        Bm = [x.to(dev) for x in inp["W"]]
        Y = [torch.empty(M, N // R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        plan = B.fo_plan("gemm_a2a", R, M, N, K)
    elif w.op == "gemm_ar":
        R, M, K, N = w.R, d["M"], d["K"], d["N"]
        A = [x.to(dev) for x in inp["X"]]
        Bm = [x.to(dev) for x in inp["W"]]
        Y = [torch.empty(M, N, dtype=torch.float32, device=dev) for _ in range(R)]
        plan = B.fo_plan("gemm_ar", R, M, N, K * R)
    elif w.op == "ag_gemm":
        R, M, K, Nr = w.R, d["M"], d["K"], d["N"]
        A = [x.to(dev) for x in inp["X"]]
        Bm = [x.to(dev) for x in inp["W"]]
        Y = [torch.empty(M, Nr, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        plan = B.fo_plan("ag_gemm", R, M, Nr * R, K)
    else:
        R, T, M, N = w.R, d["T"], d["M"], d["N"]
        A = [x.to(dev) for x in inp["X"]]
        Bm = [x.to(dev) for x in inp["dY"]]
        Y = [torch.empty(M // R, N, dtype=torch.float32, device=dev) for _ in range(R)]
        plan = B.fo_plan("dp_grad_rs", R, M, N, T)
    ws = torch.empty(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    B.fo_workspace_init(plan, ws)

    def launch(stream):
        if w.op == "gemm_a2a":
            B.fo_gemm_a2a(plan, A, Bm, Y, ws, stream)
        elif w.op == "gemm_ar":
            B.fo_gemm_ar(plan, A, Bm, Y, ws, stream)
        elif w.op == "ag_gemm":
            B.fo_ag_gemm(plan, A, Bm, Y, None, ws, stream)
        else:
            B.fo_dp_grad_rs(plan, A, Bm, Y, ws, stream)

    return inp, A, Bm, Y, plan, ws, launch


ATTN_WORKLOAD = "attn_rs_causal_r8_t8192_heads32_h4096"


def _attn_setup(B, dev, R=8, T=8192, heads=4, H=4096, causal=True, seed=12):
    """Query-split attention + output projection at the Llama-like layer's
    attention shape: 8192 tokens over R = 8 ranks, 4 heads of 128 per rank
    (32 heads), H = 4096; Q, K, V ~ N(0, 1), Wo ~ N(0, 0.02), bf16."""
    import torch
    g = torch.Generator().manual_seed(seed)
    w = heads * 128

    def draw(shape, std):
        return (torch.randn(shape, generator=g) * std).to(torch.bfloat16).to(dev)

    Q = [draw((T, w), 1.0) for _ in range(R)]
    K = [draw((T, w), 1.0) for _ in range(R)]
    V = [draw((T, w), 1.0) for _ in range(R)]
    Wo = [draw((w, H), 0.02) for _ in range(R)]
    O = [torch.empty(T, w, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    Y = [torch.empty(T // R, H, dtype=torch.float32, device=dev) for _ in range(R)]
    plan = B.fo_plan("gemm_rs", R, T, H, R * w)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    pplan = B.fo_plan("gemm_rs", R, T, H, R * w)
    pws = torch.zeros(B.fo_workspace_size(pplan), dtype=torch.uint8, device=dev)
    attn_flops = R * heads * 2.0 * 2.0 * T * T * 128 * (0.5 if causal else 1.0)
    proj_flops = 2.0 * T * H * R * w
    return {"plan": plan, "ws": ws, "attn_flops": attn_flops, "proj_flops": proj_flops,
            "flops": attn_flops + proj_flops, "heads": heads, "causal": causal,
            "Q": Q, "K": K, "V": V, "Wo": Wo, "O": O, "Y": Y,
            "mk_plan": lambda: B.fo_plan("gemm_rs", R, T, H, R * w),
            "call": lambda s: B.fo_attn_rs(plan, Q, K, V, Wo, O, Y, heads, causal, ws, s),
            "attn": lambda s: B.fo_attention(plan, Q, K, V, O, heads, causal, ws, s),
            "attn_noncausal": lambda s: B.fo_attention(plan, Q, K, V, O, heads, False, ws, s),
            "attn_noncausal_flops": attn_flops / (0.5 if causal else 1.0),
            "proj": lambda s: B.fo_gemm_rs(pplan, O, Wo, Y, pws, s)}


def measure_other_workloads(B, dev, stream, iters=20):
    """Short timed loops of the all-gather GEMM (QKV, R = 4), the DP
    gradient (R = 8), the all-to-all projection (R = 8), the fused
    all-reduce (R = 8), the query-split attention with its projection and
    the TP-SP layer (R = 8, forward + backward), on the
    device that times the default line: per workload the mean CUDA-event
    time per launch (per step for the layer), TFLOP/s, the fraction of the
    measured burst bf16 peak (each loop lasts well under a quarter second),
    algorithmic HBM bytes and GB/s, and the ncu DRAM traffic per launch when
    the committed capture matches the kernel source."""
    import torch

    from ag_gemm_gb300.inputs import WORKLOADS
    from ag_gemm_gb300.layer import LayerShape, TpspLayerProjections
    peaks, peak_src = load_peaks()
    burst = float(peaks["bf16_tflops"])
    out = {}
    for name in ("ag_gemm_qkv_r4_s4096_h4096_n3072", "dp_grad_rs_r8_t4096_4096x4096",
                 "gemm_a2a_qkv_r8_t8192_h4096_n12288", "gemm_ar_r8_t8192_k1792_n4096"):
        w = WORKLOADS[name]
        inp, A, Bm, Y, plan, ws, launch = _op_setup(B, w, dev)
        for _ in range(5):
            launch(stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        torch.cuda.synchronize(dev)
        for a, b in ev:
            a.record(stream)
            launch(stream)
            b.record(stream)
        torch.cuda.synchronize(dev)
        code, info = B.fo_status_query(plan, ws, stream)
        if code != 0:
            raise RuntimeError(f"device status {code} {info} ({name})")
        ms = sum(a.elapsed_time(b) for a, b in ev) / iters
        tf = w.flops() / (ms * 1e-3) / 1e12
        traffic = profiled_traffic(name)
        out[name] = {"ms": ms, "tflops": tf, "frac_of_burst_peak": tf / burst, "launches": iters,
                     "traffic": traffic, "hbm": hbm_summary(w, ms, traffic, peaks)}
        if w.op == "gemm_a2a":
            out[name].update(a2a_baselines(B, plan, A, Bm, Y, stream, dev, w.flops(), ms))
        del inp, A, Bm, Y, ws
        torch.cuda.empty_cache()
    # Query-split attention with its output projection (causal, the layer's
    # attention shape): the whole call, the attention launch alone
    # (fo_attention) and the projection alone.
    a = _attn_setup(B, dev)
    for _ in range(3):
        a["call"](stream)
    t_all = _time(lambda: a["call"](stream), stream, iters=10)
    t_attn = _time(lambda: a["attn"](stream), stream, iters=10)
    t_proj = _time(lambda: a["proj"](stream), stream, iters=10)
    code, info = B.fo_status_query(a["plan"], a["ws"], stream)
    if code != 0:
        raise RuntimeError(f"device status {code} {info} (attention)")
    out[ATTN_WORKLOAD] = {"ms": t_all, "tflops": a["flops"] / t_all / 1e9,
                          "frac_of_burst_peak": a["flops"] / t_all / 1e9 / burst,
                          "attention_ms": t_attn, "attention_tflops": a["attn_flops"] / t_attn / 1e9,
                          "attention_frac_of_burst_peak": a["attn_flops"] / t_attn / 1e9 / burst,
                          "attention_traffic": profiled_traffic(ATTN_WORKLOAD, ATTN_SOURCES, "attention"),
                          "projection_ms": t_proj, "projection_tflops": a["proj_flops"] / t_proj / 1e9,
                          "launches": 2, "flops": a["flops"],
                          "flops_note": "causal attention counts the lower triangle: 2 x 2 x T x T x 128 / 2 per head"}
    del a
    torch.cuda.empty_cache()
    shape = LayerShape(R=8, T=8192, H=4096, F=14336)
    L = TpspLayerProjections(shape, device=dev, seed=4)
    for _ in range(3):
        L.forward(stream)
        L.backward(stream)
    steps = 5
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    L.launches = 0
    a.record(stream)
    for _ in range(steps):
        L.forward(stream)
        L.backward(stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    if any(L.status()):
        raise RuntimeError(f"device status {L.status()} (layer)")
    ms = a.elapsed_time(b) / steps
    tf = shape.flops()["total"] / (ms * 1e-3) / 1e12
    out[LAYER_WORKLOAD] = {"ms": ms, "tflops": tf, "frac_of_burst_peak": tf / burst,
                           "launches": L.launches, "steps": steps, "traffic": None}
    del L
    torch.cuda.empty_cache()
    out["peak_source"] = f"bf16_tflops (burst), {peak_src}"
    return out


def a2a_baselines(B, plan, X, W, Y, stream, dev, flops, fused_ms):
    """Same-GPU comparisons of the fused all-to-all projection: each rank's
    whole projection by cuBLAS (torch.matmul, bf16 out), and the unfused
    path (those GEMMs, then the separate all-to-all copy kernel)."""
    import torch
    R = len(X)
    P = [torch.empty(X[0].shape[0], W[0].shape[1], dtype=torch.bfloat16, device=dev) for _ in range(R)]

    def cublas():
        for r in range(R):
            torch.matmul(X[r], W[r], out=P[r])

    def unfused():
        cublas()
        B.fo_all_to_all_copy(plan, P, Y, stream)

    cub = _time(cublas, stream)
    unf = _time(unfused, stream)
    copy = _time(lambda: B.fo_all_to_all_copy(plan, P, Y, stream), stream)
    del P
    torch.cuda.empty_cache()
    return {"cublas_matmul_ms": cub, "cublas_matmul_tflops": flops / cub / 1e9,
            "unfused_ms": unf, "unfused_tflops": flops / unf / 1e9, "unfused_copy_kernel_ms": copy,
            "latency_reduction_vs_unfused_pct": 100.0 * (1.0 - fused_ms / unf)}


def run_other_op(args, w, dev, world, rank):
    """Timed loop of the AG-GEMM, A2A, AR or DP-grad-RS workloads (same
    timing rules as the default line; no comparison legs)."""
    import torch
    import torch.distributed as dist

    from ag_gemm_gb300 import binding as B
    d = w.dims
    stream = torch.cuda.current_stream(dev)
    inp, A, Bm, Y, plan, ws, launch = _op_setup(B, w, dev)
    if w.op in ("ag_gemm", "gemm_a2a", "gemm_ar"):
        R, M, K, Nr = w.R, d["M"], d["K"], d["N"]
    else:
        R, T, M, N = w.R, d["T"], d["M"], d["N"]

    def step():
        launch(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    # Only this op's launches, back to back: the region's event time over
    # the step count is the average launch duration.
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(_smi_id(dev)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        clk.mark("t0")
        t0.record(stream)
        for i in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("t1")
    code, info = B.fo_status_query(plan, ws, stream)
    if code != 0:
        raise RuntimeError(f"device status {code} {info}")
    elapsed_ms = t0.elapsed_time(t1)
    if w.op == "gemm_a2a":
        e2e = measure_e2e(B, lambda: B.fo_plan("gemm_a2a", R, M, Nr, K),
                          lambda p, din, dout, ws_, s_: B.fo_gemm_a2a(p, din[0], din[1], dout, ws_, s_),
                          [inp["X"], inp["W"]], [A, Bm], Y, dev, stream, world, w.flops(),
                          max(4, min(args.steps, 12)))
    elif w.op == "gemm_ar":
        e2e = measure_e2e(B, lambda: B.fo_plan("gemm_ar", R, M, Nr, K * R),
                          lambda p, din, dout, ws_, s_: B.fo_gemm_ar(p, din[0], din[1], dout, ws_, s_),
                          [inp["X"], inp["W"]], [A, Bm], Y, dev, stream, world, w.flops(),
                          max(4, min(args.steps, 12)))
    elif w.op == "ag_gemm":
        e2e = measure_e2e(B, lambda: B.fo_plan("ag_gemm", R, M, Nr * R, K),
                          lambda p, din, dout, ws_, s_: B.fo_ag_gemm(p, din[0], din[1], dout, None, ws_, s_),
                          [inp["X"], inp["W"]], [A, Bm], Y, dev, stream, world, w.flops(),
                          max(4, min(args.steps, 12)))
    else:
        e2e = measure_e2e(B, lambda: B.fo_plan("dp_grad_rs", R, M, N, T),
                          lambda p, din, dout, ws_, s_: B.fo_dp_grad_rs(p, din[0], din[1], dout, ws_, s_),
                          [inp["X"], inp["dY"]], [A, Bm], Y, dev, stream, world, w.flops(),
                          max(4, min(args.steps, 12)))
    kernel_ms = elapsed_ms / args.steps
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    flops = w.flops()
    peaks, peak_src = load_peaks()
    sustained = elapsed_ms >= 250.0
    peak = float(peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(w.name),
                     "peak_source": ("bf16_tflops_sustained" if sustained else "bf16_tflops (burst)") + ", " + peak_src},
        "hbm": hbm_summary(w, kernel_ms, profiled_traffic(w.name), peaks),
        "e2e": e2e,
        "gpu_launches": args.steps * B.fo_plan_last_launches(plan),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        tf, desc = oracle_sample(w, oracle_inputs(w))
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line))
    return 0


def _loop_ms(fn, stream, dev, iters):
    """Mean CUDA-event time of one fn(stream) call over `iters` back-to-back
    calls, after three untimed ones."""
    import torch
    for _ in range(3):
        fn(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    torch.cuda.synchronize(dev)
    for a, b in ev:
        a.record(stream)
        fn(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / iters


def run_attn(args, dev, world, rank):
    """One step = one fo_attn_rs call: query-split causal attention of 32
    heads over 8192 tokens (R = 8), then the fused output projection +
    reduce-scatter (two launches). The roofline is the attention kernel's,
    timed alone through fo_attention; the projection is timed alone too."""
    import torch
    import torch.distributed as dist

    from ag_gemm_gb300 import binding as B
    a = _attn_setup(B, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        a["call"](stream)
    steps = max(1, min(args.steps, 500))
    with ClockSampler(_smi_id(dev)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        clk.mark("t0")
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            a["call"](stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("t1")
        attn_ms = _loop_ms(a["attn"], stream, dev, steps)
        proj_ms = _loop_ms(a["proj"], stream, dev, steps)
        full_ms = _loop_ms(a["attn_noncausal"], stream, dev, steps)
    code, info = B.fo_status_query(a["plan"], a["ws"], stream)
    if code != 0:
        raise RuntimeError(f"device status {code} {info}")
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / steps
    peaks, peak_src = load_peaks()
    sustained = ms * steps >= 250.0
    peak = float(peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
    burst = float(peaks["bf16_tflops"])
    value = world * a["flops"] / (ms * 1e-3) / 1e12
    attn_tf = a["attn_flops"] / (attn_ms * 1e-3) / 1e12
    proj_tf = a["proj_flops"] / (proj_ms * 1e-3) / 1e12
    heads, causal, O = a["heads"], a["causal"], a["O"]
    e2e = measure_e2e(B, a["mk_plan"],
                      lambda p, din, dout, ws_, s_: B.fo_attn_rs(p, din[0], din[1], din[2], din[3], O, dout,
                                                                 heads, causal, ws_, s_),
                      [[t.cpu() for t in a[n]] for n in ("Q", "K", "V", "Wo")],
                      [a["Q"], a["K"], a["V"], a["Wo"]], a["Y"], dev, stream, world, a["flops"],
                      max(4, min(args.steps, 12)))
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": ATTN_WORKLOAD, "R": 8, "tokens": 8192, "heads": 32, "head_dim": 128,
                   "hidden": 4096, "causal": True,
                   "step": "query-split attention + fused output projection and reduce-scatter (2 launches)",
                   "l2": "no flush: 470 MB of operands and outputs per step"},
        # The dominant kernel: the attention launch, timed alone (burst
        # peak: one loop of `steps` launches lasts well under a second).
        "roofline": {"bound": "tensor", "achieved": attn_tf, "peak": burst, "unit": "TFLOP/s",
                     "frac": attn_tf / burst, "traffic": profiled_traffic(ATTN_WORKLOAD, ATTN_SOURCES, "attention"),
                     "kernel": "fo_attn_kernel", "ms": attn_ms,
                     "peak_source": "bf16_tflops (burst), " + peak_src},
        "kernels": {"attention": {"ms": attn_ms, "tflops": attn_tf, "frac_of_burst_peak": attn_tf / burst,
                                  "flops": a["attn_flops"]},
                    "projection_rs": {"ms": proj_ms, "tflops": proj_tf, "frac_of_burst_peak": proj_tf / burst,
                                      "flops": a["proj_flops"]},
                    # The same launch without the causal mask (every query
                    # sees every key): uniform items, twice the work.
                    "attention_noncausal": {"ms": full_ms,
                                            "tflops": a["attn_noncausal_flops"] / (full_ms * 1e-3) / 1e12,
                                            "frac_of_burst_peak": a["attn_noncausal_flops"] / (full_ms * 1e-3) / 1e12 / burst,
                                            "flops": a["attn_noncausal_flops"]},
                    "step_frac_of_peak": value / world / peak,
                    "step_peak_source": ("bf16_tflops_sustained" if sustained else "bf16_tflops (burst)")},
        "e2e": e2e,
        "gpu_launches": 2 * steps,
        "clocks": clk.summary(),
        "flops_per_step": a["flops"],
    }
    if rank == 0:
        print(json.dumps(line))
    return 0


def run_layer(args, dev, world, rank):
    """One step = forward + backward of the projections of one TP-SP layer
    (R = 8, 8192 tokens, hidden 4096, FFN 14336): 4 fused collective GEMMs
    forward, 4 fused collective GEMMs + 4 weight-gradient GEMMs backward."""
    import torch
    import torch.distributed as dist

    from ag_gemm_gb300.layer import LayerShape, TpspLayerProjections
    shape = LayerShape(R=8, T=8192, H=4096, F=14336)
    L = TpspLayerProjections(shape, device=dev, seed=4)
    flops = shape.flops()["total"]
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 3)):
        L.forward(stream)
        L.backward(stream)
    torch.cuda.synchronize(dev)
    if any(L.status()):
        raise RuntimeError(f"device status {L.status()}")
    L.launches = 0
    steps = max(1, min(args.steps, 200))
    with ClockSampler(_smi_id(dev)) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        clk.mark("t0")
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            L.forward(stream)
            L.backward(stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark("t1")
    ms = max_over_ranks(a.elapsed_time(b), world, dev) / steps
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops_sustained"])
    value = world * flops / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": LAYER_WORKLOAD, "R": 8, "tokens": 8192, "hidden": 4096, "ffn": 14336,
                   "heads": 32, "step": "forward + backward projections (attention core, SwiGLU, norms excluded)",
                   "l2": "no flush: several GB of operands per step"},
        "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / world / peak, "traffic": None,
                     "peak_source": f"bf16_tflops_sustained, {peak_src}"},
        "gpu_launches": L.launches,
        "clocks": clk.summary(),
        "flops_per_step": flops,
    }
    if rank == 0:
        print(json.dumps(line))
    return 0


def run_sweep(args):
    """NEXT-style sweeps, one JSON line: the MLP block of a TP layer (AG-GEMM
    up|gate, then GEMM-RS down; hidden 4096, FFN 14336, R = 4) over sequence
    lengths, fused versus the unfused same-GPU path (gather copy + GEMMs;
    GEMMs to partials + reduce kernel), plus the data-slicing order."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from ag_gemm_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    R, H, F = 4, 4096, 14336
    peaks, _ = load_peaks()
    burst, hbm_peak = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    seqs = [int(x) for x in args.sweep_seqs.split(",")]
    g = torch.Generator().manual_seed(6)
    rows = []
    for T in seqs:
        x = [(torch.randn(T // R, H, generator=g)).bfloat16().to(dev) for _ in range(R)]
        Wug = [(torch.randn(H, 2 * F // R, generator=g) * 0.02).bfloat16().to(dev) for _ in range(R)]
        act = [(torch.randn(T, F // R, generator=g)).bfloat16().to(dev) for _ in range(R)]
        Wd = [(torch.randn(F // R, H, generator=g) * 0.02).bfloat16().to(dev) for _ in range(R)]
        y_ug = [torch.empty(T, 2 * F // R, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        y = [torch.empty(T // R, H, device=dev) for _ in range(R)]
        p_ug = B.fo_plan("ag_gemm", R, T, 2 * F, H)
        p_d = B.fo_plan("gemm_rs", R, T, H, F)
        p_ds = B.fo_plan("gemm_rs", R, T, H, F, sched="sliced")
        ws = {k: torch.zeros(B.fo_workspace_size(pp), dtype=torch.uint8, device=dev)
              for k, pp in (("ug", p_ug), ("d", p_d), ("ds", p_ds))}

        def fused():
            B.fo_ag_gemm(p_ug, x, Wug, y_ug, None, ws["ug"], stream)
            B.fo_gemm_rs(p_d, act, Wd, y, ws["d"], stream)

        def sliced():
            B.fo_ag_gemm(p_ug, x, Wug, y_ug, None, ws["ug"], stream)
            B.fo_gemm_rs(p_ds, act, Wd, y, ws["ds"], stream)

        G = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(R)]
        P = [torch.empty(T, H, device=dev) for _ in range(R)]
        p_one = [B.fo_plan("ag_gemm", 1, T, 2 * F // R, H) for _ in range(R)]
        ws1 = [torch.zeros(B.fo_workspace_size(pp), dtype=torch.uint8, device=dev) for pp in p_one]
        p_part = B.fo_plan("gemm_rs", R, T, H, F)   # own plan: its launch parameters stay cached

        def unfused():
            B.fo_all_gather_copy(p_ug, x, G, stream)
            for r in range(R):
                B.fo_ag_gemm(p_one[r], [G[r]], [Wug[r]], [y_ug[r]], None, ws1[r], stream)
            B.fo_gemm_partials(p_part, act, Wd, P, ws["d"], stream)
            B.fo_reduce_scatter_f32(p_part, P, y, stream)

        flops = 2.0 * T * H * 2 * F + 2.0 * T * F * H
        t_f, t_s, t_u = _time(fused, stream), _time(sliced, stream), _time(unfused, stream)
        # HBM roofline of the fused pair: bytes each launch must move at
        # least (operands once, outputs once, the RS partials to their owners
        # and back), and the operand bytes the per-chunk decomposition pulls
        # from L2 into the SMs (every chunk task reads all of its rank's
        # weight, so the weights cross R times; the X chunks once each).
        w_ug, w_d = H * 2 * F * 2.0, F * H * 2.0                  # all ranks' weights
        hbm_bytes = (T * H * 2.0 + w_ug + T * 2 * F * 2.0) + \
                    (T * F * 2.0 + w_d + 2.0 * (R - 1) * T * H * 4 + T * H * 4.0)
        l2_operand_bytes = R * (w_ug + w_d) + R * T * H * 2.0 + T * F * 2.0
        rows.append({"seq": T, "fused_ms": t_f, "sliced_ms": t_s, "unfused_ms": t_u,
                     "fused_tflops": flops / t_f / 1e9,
                     "frac_of_burst_peak": flops / t_f / 1e9 / burst,
                     "hbm_algorithmic_bytes": hbm_bytes,
                     "hbm_frac": hbm_bytes / (t_f * 1e-3) / 1e9 / hbm_peak,
                     "l2_operand_bytes": l2_operand_bytes,
                     "l2_operand_gbs": l2_operand_bytes / (t_f * 1e-3) / 1e9,
                     "latency_reduction_vs_unfused_pct": 100.0 * (t_u - t_f) / t_u,
                     "sliced_reduction_vs_unfused_pct": 100.0 * (t_u - t_s) / t_u})
        del x, Wug, act, Wd, y_ug, y, G, P, ws, ws1
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "mlp_block_seq", "R": R, "hidden": H, "ffn": F, "rows": rows}))
    return 0


def run_single_gemm(args):
    """One rank's GEMM (8192 x 4096 x K) through the fused kernel with a
    bf16 output (R = 1 all-gather plan) and an fp32 output (R = 1 partials
    control), next to cuBLAS bf16 on the same operands; one JSON line of
    TFLOP/s. The inputs stay in L2, so this isolates the kernel's main loop
    and epilogue from HBM and from the R-rank schedule."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from ag_gemm_gb300 import binding as B
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    M, N = 8192, 4096
    g = torch.Generator().manual_seed(2)
    rows = []
    for K in (1792, 4096):
        X = torch.randn(M, K, generator=g).bfloat16().to(dev)
        W = (torch.randn(K, N, generator=g) * 0.02).bfloat16().to(dev)
        y16 = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        y32 = torch.empty(M, N, device=dev)
        pa = B.fo_plan("ag_gemm", 1, M, N, K)
        wa = torch.zeros(B.fo_workspace_size(pa), dtype=torch.uint8, device=dev)
        pp = B.fo_plan("gemm_rs", 1, M, N, K)
        wp = torch.zeros(B.fo_workspace_size(pp), dtype=torch.uint8, device=dev)
        flops = 2.0 * M * N * K
        t_cub = _time(lambda: torch.matmul(X, W, out=y16), stream, iters=args.steps, warm=args.warmup)
        t_bf = _time(lambda: B.fo_ag_gemm(pa, [X], [W], [y16], None, wa, stream), stream, iters=args.steps,
                     warm=args.warmup)
        t_f32 = _time(lambda: B.fo_gemm_partials(pp, [X], [W], [y32], wp, stream), stream, iters=args.steps,
                      warm=args.warmup)
        rows.append({"K": K, "cublas_bf16_tflops": flops / t_cub / 1e9, "fused_bf16_out_tflops": flops / t_bf / 1e9,
                     "fused_f32_out_tflops": flops / t_f32 / 1e9})
        del X, W, y16, y32, wa, wp
        torch.cuda.empty_cache()
    print(json.dumps({"single_gemm": {"M": M, "N": N}, "rows": rows}))
    return 0


def _smi_id(dev) -> str:
    """nvidia-smi selector of a torch device (its UUID when torch exposes it)."""
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev.index or 0)


def _time(fn, stream, iters=10, warm=2):
    import torch
    for _ in range(warm):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(iters):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def traced_tail_us(B, desc, call, stream, dev, reps=5):
    """Median over `reps` traced launches of the exposed tail (time the last
    transfer ran past the last MMA) and of the launch span, in us, from the
    kernel's own %globaltimer stamps."""
    import torch
    desc = dict(desc)
    op, R, M, N, K = (desc.pop(k) for k in ("op", "R", "M", "N", "K"))
    plan = B.fo_plan(op, R, M, N, K, trace=True, **desc)
    ws = torch.zeros(B.fo_workspace_size(plan), dtype=torch.uint8, device=dev)
    call(plan, ws)
    tails, spans = [], []
    for _ in range(reps):
        call(plan, ws)
        s = B.trace_summary(B.fo_trace_query(plan, ws, stream))
        tails.append(s["exposed_tail_ns"] / 1e3)
        spans.append(s["span_ns"] / 1e3)
    del ws
    return {"tail_us": sorted(tails)[reps // 2], "span_us": sorted(spans)[reps // 2]}


class DataSlicing:
    """The data-slicing baseline of the pages ([GS] "Technical Summary" §1,
    Existing Solutions): the GEMM-RS cut into S row slices of M/S rows. Each
    slice's GEMM (all R ranks' rows of that slice, one launch, fp32 partials)
    runs on the launching stream; that slice's reduce-scatter (a separate
    kernel) runs on a side stream once the slice's GEMM is done, overlapping
    the next slice's GEMM. The last slice's reduce-scatter has no compute
    left to hide behind: it is the tail. Rank d's output holds, for each
    slice j in order, its M/(S*R) rows of that slice (slicing changes which
    rows a rank owns; the sums are the same)."""

    def __init__(self, B, R, M, N, Kr, S, dev):
        import torch
        if M % (S * R):
            raise ValueError("M must split into S slices of R chunks")
        self.B, self.R, self.S, self.Ms = B, R, S, M // S
        tile = "auto" if self.Ms // R >= 256 else "single"
        # One plan per slice: each keeps its own cached launch parameters.
        self.plans = [B.fo_plan("gemm_rs", R, self.Ms, N, Kr * R, tile_config=tile) for _ in range(S)]
        self.ws = [torch.zeros(B.fo_workspace_size(p), dtype=torch.uint8, device=dev) for p in self.plans]
        self.P = [torch.empty(M, N, dtype=torch.float32, device=dev) for _ in range(R)]
        self.side = torch.cuda.Stream(dev)

    def __call__(self, X, W, Y, stream):
        import torch
        B, R, Ms = self.B, self.R, self.Ms
        start = torch.cuda.Event()
        start.record(stream)
        self.side.wait_event(start)       # the previous call's readers of P are done
        for j, plan in enumerate(self.plans):
            Ps = [p[j * Ms:(j + 1) * Ms] for p in self.P]
            B.fo_gemm_partials(plan, [x[j * Ms:(j + 1) * Ms] for x in X], W, Ps, self.ws[j], stream)
            ready = torch.cuda.Event()
            ready.record(stream)
            self.side.wait_event(ready)
            B.fo_reduce_scatter_f32(plan, Ps, [y[j * Ms // R:(j + 1) * Ms // R] for y in Y], self.side)
        done = torch.cuda.Event()
        done.record(self.side)
        stream.wait_event(done)


def slicing_sweep(B, X, W, Y, stream, dev, fused, pure, unfused, counts=(1, 2, 4, 8, 16)):
    """Data slicing over chunk counts against the fused launch, with the
    pages' measure ([GS] §4): the share of the serial path's communication
    overhead (unfused minus the pure GEMM) that a method removes."""
    import torch
    R, (M, Kr), N = len(X), X[0].shape, W[0].shape[1]
    overhead = unfused - pure

    def reduction(t):
        return 100.0 * (1.0 - (t - pure) / overhead) if overhead > 0 else None

    rows = []
    for S in counts:
        if M % (S * R):
            continue
        ds = DataSlicing(B, R, M, N, Kr, S, dev)
        t = _time(lambda: ds(X, W, Y, stream), stream)
        rows.append({"chunks": S, "ms": t, "overhead_reduction_pct": reduction(t)})
        del ds
        torch.cuda.empty_cache()
    return {"rows": rows, "fused_overhead_reduction_pct": reduction(fused),
            "pure_gemm_ms": pure, "unfused_serial_ms": unfused}


def measure_extras(B, plan, X, W, Y, ws, stream, flops, dev):
    """Same-GPU comparisons: pure-GEMM control (no transfer), unfused
    (GEMM to per-rank partials, then a separate reduce kernel), cuBLAS with
    bf16 and with fp32 output."""
    import torch
    R = len(X)
    M, N = X[0].shape[0], W[0].shape[1]
    fused = _time(lambda: B.fo_gemm_rs(plan, X, W, Y, ws, stream), stream)
    P = [torch.empty(M, N, dtype=torch.float32, device=dev) for _ in range(R)]
    pure = _time(lambda: B.fo_gemm_partials(plan, X, W, P, ws, stream), stream)
    red = _time(lambda: B.fo_reduce_scatter_f32(plan, P, Y, stream), stream)

    def unfused():
        B.fo_gemm_partials(plan, X, W, P, ws, stream)
        B.fo_reduce_scatter_f32(plan, P, Y, stream)

    unf = _time(unfused, stream)

    def cublas():
        for r in range(R):
            torch.matmul(X[r], W[r])

    cub = _time(cublas, stream)

    # The same GEMMs by cuBLAS with fp32 output (bf16 inputs, fp32
    # accumulate): the output bytes the fused kernel's partials carry.
    def cublas_f32():
        for r in range(R):
            torch.mm(X[r], W[r], out_dtype=torch.float32, out=P[r])

    try:
        cub32 = _time(cublas_f32, stream)
    except (TypeError, RuntimeError):   # a torch without mm's out_dtype
        cub32 = None
    del P
    torch.cuda.empty_cache()
    # Schedule ablation: the data-slicing order (every rank on slice s at
    # step s) instead of the rank-adaptive one, same kernel otherwise.
    sl_plan = B.fo_plan("gemm_rs", R, M, N, X[0].shape[1] * R, sched="sliced")
    sl_ws = torch.zeros(B.fo_workspace_size(sl_plan), dtype=torch.uint8, device=dev)
    sliced = _time(lambda: B.fo_gemm_rs(sl_plan, X, W, Y, sl_ws, stream), stream)
    # Single-CTA 128 x 256 tiles instead of CTA-pair 256 x 256 tiles.
    one_plan = B.fo_plan("gemm_rs", R, M, N, X[0].shape[1] * R, tile_config="single")
    one_ws = torch.zeros(B.fo_workspace_size(one_plan), dtype=torch.uint8, device=dev)
    single = _time(lambda: B.fo_gemm_rs(one_plan, X, W, Y, one_ws, stream), stream)
    del one_ws, sl_ws
    # The ring reduce-scatter (running sums forwarded rank to rank) and the
    # direct algorithm's in-order (deterministic) adds, same kernel order.
    ring_plan = B.fo_plan("gemm_rs", R, M, N, X[0].shape[1] * R, rs_algo="ring")
    ring_ws = torch.zeros(B.fo_workspace_size(ring_plan), dtype=torch.uint8, device=dev)
    ring = _time(lambda: B.fo_gemm_rs(ring_plan, X, W, Y, ring_ws, stream), stream)
    del ring_ws
    det_plan = B.fo_plan("gemm_rs", R, M, N, X[0].shape[1] * R, deterministic=True)
    det_ws = torch.zeros(B.fo_workspace_size(det_plan), dtype=torch.uint8, device=dev)
    det = _time(lambda: B.fo_gemm_rs(det_plan, X, W, Y, det_ws, stream), stream)
    del det_ws
    torch.cuda.empty_cache()
    tails = {}
    for name, kw in (("rank_adaptive", {}), ("sliced", dict(sched="sliced"))):
        tails[name] = traced_tail_us(B, dict(op="gemm_rs", R=R, M=M, N=N, K=X[0].shape[1] * R, **kw),
                                     lambda p, w: B.fo_gemm_rs(p, X, W, Y, w, stream), stream, dev)
    slicing = slicing_sweep(B, X, W, Y, stream, dev, fused, pure, unf)
    return {
        "data_slicing": slicing,
        "exposed_tail_us": tails,
        "ring_rs_ms": ring, "ring_rs_tflops": flops / ring / 1e9,
        "direct_in_order_adds_ms": det, "direct_in_order_adds_tflops": flops / det / 1e9,
        "sliced_schedule_ms": sliced, "sliced_schedule_tflops": flops / sliced / 1e9,
        "single_cta_tiles_ms": single, "single_cta_tiles_tflops": flops / single / 1e9,
        "fused_ms": fused, "fused_tflops": flops / fused / 1e9,
        "pure_gemm_control_ms": pure, "pure_gemm_control_tflops": flops / pure / 1e9,
        "exposed_move_pct": 100.0 * (fused - pure) / pure,
        "unfused_ms": unf, "unfused_tflops": flops / unf / 1e9, "unfused_reduce_kernel_ms": red,
        "cublas_matmul_bf16_out_ms": cub, "cublas_matmul_tflops": flops / cub / 1e9,
        "cublas_matmul_fp32_out_ms": cub32,
        "cublas_matmul_fp32_out_tflops": flops / cub32 / 1e9 if cub32 else None,
        "fused_over_cublas_fp32_out": fused / cub32 if cub32 else None,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true", help="skip the control/unfused/cuBLAS comparisons")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: MLP-block sweep over --sweep-seqs (one JSON line)")
    ap.add_argument("--sweep-seqs", default="128,512,1024,2048,4096,8192,16384")
    ap.add_argument("--single-gemm", action="store_true",
                    help="instead of the bench line: one rank's GEMM, fused kernel against cuBLAS (one JSON line)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the fused kernel from an ncu capture of this build")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.single_gemm:
        return run_single_gemm(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
