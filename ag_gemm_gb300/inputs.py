"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers; it holds none of the method's
arithmetic. Every generator uses one CPU ``torch.Generator(seed)`` and draws
the tensors in a fixed order: X_0..X_{R-1}, then W_0..W_{R-1} (or dY_0..).

Value recipes (the pages' workloads are LLM layers with d_model 4096, TP 4 and
sequence 1K-16K; the configurations below are synthetic stand-ins):

* ``"int"``   : integers uniform in [-4, 4] (every fp32 partial sum is exact);
* ``"randn"`` : activations / upstream gradients ~ N(0, 1), weights ~ N(0, w_std).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List

import torch

_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _draw(g: torch.Generator, shape, mode: str, std: float, dtype: str) -> torch.Tensor:
    if mode == "int":
        t = torch.randint(-4, 5, shape, generator=g, dtype=torch.int32).to(torch.float32)
    elif mode == "randn":
        t = torch.randn(shape, generator=g, dtype=torch.float32) * std
    else:
        raise ValueError(f"unknown mode {mode!r}")
    return t.to(_DT[dtype])


def gemm_rs_inputs(R: int, M: int, K: int, N: int, *, dtype="bf16", mode="randn",
                   seed=0, w_std=0.02, w_layout="kn") -> Dict[str, List[torch.Tensor]]:
    """X_r [M, K] (K = per-rank reduction size), W_r [K, N] (``w_layout="kn"``)
    or its transpose stored [N, K] (``"nk"``, the nn.Linear weight layout)."""
    g = torch.Generator().manual_seed(seed)
    X = [_draw(g, (M, K), mode, 1.0, dtype) for _ in range(R)]
    W = [_draw(g, (K, N), mode, w_std, dtype) for _ in range(R)]
    if w_layout == "nk":
        W = [w.t().contiguous() for w in W]
    return {"X": X, "W": W}


def ag_gemm_inputs(R: int, M: int, K: int, N: int, *, dtype="bf16", mode="randn",
                   seed=1, w_std=0.02, w_layout="kn") -> Dict[str, List[torch.Tensor]]:
    """X_r [M/R, K] (row shard of the sequence), W_r [K, N] with N the per-rank
    output width (or [N, K] for ``w_layout="nk"``)."""
    if M % R:
        raise ValueError("M must be divisible by R")
    g = torch.Generator().manual_seed(seed)
    X = [_draw(g, (M // R, K), mode, 1.0, dtype) for _ in range(R)]
    W = [_draw(g, (K, N), mode, w_std, dtype) for _ in range(R)]
    if w_layout == "nk":
        W = [w.t().contiguous() for w in W]
    return {"X": X, "W": W}


def dp_grad_inputs(R: int, T: int, M: int, N: int, *, dtype="bf16", mode="randn",
                   seed=3) -> Dict[str, List[torch.Tensor]]:
    """X_r [T, M] activations and dY_r [T, N] upstream gradients, ~N(0, 1)."""
    g = torch.Generator().manual_seed(seed)
    X = [_draw(g, (T, M), mode, 1.0, dtype) for _ in range(R)]
    dY = [_draw(g, (T, N), mode, 1.0, dtype) for _ in range(R)]
    return {"X": X, "dY": dY}


@dataclass(frozen=True)
class Workload:
    """One named workload: the op, the virtual rank count and the global sizes."""
    name: str
    op: str            # "gemm_rs" | "gemm_ar" | "ag_gemm" | "dp_grad_rs" | "gemm_a2a"
    R: int
    dims: Dict[str, int] = field(default_factory=dict)
    dtype: str = "bf16"
    mode: str = "randn"
    seed: int = 0

    def flops(self) -> float:
        d = self.dims
        if self.op in ("gemm_rs", "gemm_ar"):
            return 2.0 * self.R * d["M"] * d["N"] * d["K"]
        if self.op == "ag_gemm":
            return 2.0 * self.R * d["M"] * d["N"] * d["K"]
        if self.op == "gemm_a2a":
            return 2.0 * d["M"] * d["N"] * d["K"]
        if self.op == "dp_grad_rs":
            return 2.0 * self.R * d["M"] * d["N"] * d["T"]
        raise ValueError(self.op)

    def make(self, **kw):
        d = self.dims
        if self.op in ("gemm_rs", "gemm_ar"):
            return gemm_rs_inputs(self.R, d["M"], d["K"], d["N"], dtype=self.dtype,
                                  mode=self.mode, seed=self.seed, **kw)
        if self.op in ("ag_gemm", "gemm_a2a"):
            return ag_gemm_inputs(self.R, d["M"], d["K"], d["N"], dtype=self.dtype,
                                  mode=self.mode, seed=self.seed, **kw)
        if self.op == "dp_grad_rs":
            return dp_grad_inputs(self.R, d["T"], d["M"], d["N"], dtype=self.dtype,
                                  mode=self.mode, seed=self.seed)
        raise ValueError(self.op)


# The named workloads. Sizes are global: M rows of the RS / AR output /
# gathered sequence, K the per-rank reduction size (RS, AR) or hidden size
# (AG, A2A), N the output width per rank (AG) or total (RS, AR, A2A: all R
# head groups), T tokens (DP grad). The all-to-all draws its inputs like the all-gather: X_r
# [M/R x K], then W_r [K x N] (the whole projection on every rank).
WORKLOADS = {
    "gemm_rs_int_r2_256x512x512": Workload("gemm_rs_int_r2_256x512x512", "gemm_rs", 2,
                                           {"M": 256, "K": 512, "N": 512}, "f32", "int", 0),
    "ag_gemm_qkv_r4_s4096_h4096_n3072": Workload("ag_gemm_qkv_r4_s4096_h4096_n3072", "ag_gemm", 4,
                                                 {"M": 4096, "K": 4096, "N": 3072}, "bf16", "randn", 1),
    "gemm_rs_down_r8_t8192_k1792_n4096": Workload("gemm_rs_down_r8_t8192_k1792_n4096", "gemm_rs", 8,
                                                  {"M": 8192, "K": 1792, "N": 4096}, "bf16", "randn", 2),
    # The fused all-reduce (reduce-scatter, then every finished tile copied
    # into every rank's full output) on the down projection's shape.
    "gemm_ar_r8_t8192_k1792_n4096": Workload("gemm_ar_r8_t8192_k1792_n4096", "gemm_ar", 8,
                                             {"M": 8192, "K": 1792, "N": 4096}, "bf16", "randn", 2),
    "dp_grad_rs_r8_t4096_4096x4096": Workload("dp_grad_rs_r8_t4096_4096x4096", "dp_grad_rs", 8,
                                              {"T": 4096, "M": 4096, "N": 4096}, "bf16", "randn", 3),
    # Ulysses QKV projection of the Llama-like layer's shape: 8192 tokens
    # over R = 8, hidden 4096, Q|K|V of 32 heads (12288 columns, 4 heads of
    # 128 per rank after the all-to-all).
    "gemm_a2a_qkv_r8_t8192_h4096_n12288": Workload("gemm_a2a_qkv_r8_t8192_h4096_n12288", "gemm_a2a", 8,
                                                   {"M": 8192, "K": 4096, "N": 12288}, "bf16", "randn", 5),
}
