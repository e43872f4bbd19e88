"""The projection GEMMs of one tensor- and sequence-parallel (TP-SP)
transformer layer, forward and backward, on the fused collectives.

The pages name this use: the method is instantiated for the row- and
column-parallel projections of MLP and QKV layers (gist.science, "Technical
Summary" section 2, "Architectural Versatility"), in training forward and
backward (section 3). With R virtual ranks, a sequence of T tokens split
T/R per rank, hidden size H and FFN size F:

forward
    QKV     column-parallel: AG-GEMM      Y_qkv_r = AllGather(x) . Wqkv_r    [H x 3H/R]
    o       row-parallel:    GEMM-RS      h       = RS(attn_r . Wo_r)        [H/R x H]
    up|gate column-parallel: AG-GEMM      Y_ug_r  = AllGather(h) . Wug_r     [H x 2F/R]
    down    row-parallel:    GEMM-RS      y       = RS(act_r . Wd_r)         [F/R x H]
backward (the usual TP-SP duals; the pages do not spell them out)
    row-parallel GEMM-RS Y = RS(X_r . W_r):
        dX_r = AllGather(dY) . W_r^T          AG-GEMM, W read as [N x K]
        dW_r = X_r^T . AllGather(dY)          per-rank weight GEMM (partials)
    column-parallel AG-GEMM Y_r = AllGather(X) . W_r:
        dX   = RS(dY_r . W_r^T)               GEMM-RS, W read as [N x K]
        dW_r = AllGather(X)^T . dY_r          per-rank weight GEMM (partials)
The weight gradients of the row-parallel projections (o, down) are produced
transposed, as AllGather(dY)^T . X_r, i.e. in the nn.Linear layout
[out x in] = [H x H/R] and [H x F/R]: the per-rank GEMM then splits H rows
into R chunks of H/R rows instead of H/R or F/R rows into R chunks (64 or
224 rows for the default shape, which fill 128- and 256-row tiles poorly).
Each weight gradient contracts over all T tokens of an all-gathered
operand; it reads the R token shards where they lie, so no gathered copy
of x, h, dy or dh is written. Those shards are allocated back to back in
rank order, which the weight-gradient call reads as one tensor.

The attention core, the SwiGLU and the norms are not part of the path: their
outputs (attn_r, act_r) and upstream gradients are fixed synthetic tensors.
Every GEMM runs in the library's kernels; this module only allocates
buffers and issues the calls: 12 launches per forward + backward (4
forward collective GEMMs, 4 backward data-gradient collective GEMMs and 4
per-rank weight-gradient GEMMs).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List

import torch

from . import binding as B


@dataclass(frozen=True)
class LayerShape:
    R: int = 8
    T: int = 8192
    H: int = 4096
    F: int = 14336

    def flops(self) -> Dict[str, float]:
        T, H, F = self.T, self.H, self.F
        fwd = 2.0 * T * H * (3 * H) + 2.0 * T * H * H + 2.0 * T * H * (2 * F) + 2.0 * T * F * H
        return {"forward": fwd, "backward": 2 * fwd, "total": 3 * fwd}


def _draw(g, shape, std, device):
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16).to(device)


def _ints(g, shape, device):
    return torch.randint(-4, 5, shape, generator=g, dtype=torch.int32).to(torch.bfloat16).to(device)


class TpspLayerProjections:
    """Buffers, plans and launches for one layer's projections (R virtual ranks
    on one GPU). `mode="randn"` draws weights ~N(0, 0.02) and activations /
    gradients ~N(0, 1); `mode="int"` draws integers in [-4, 4] so every sum
    is exact in fp32.

    The weight gradients after an all-gather GEMM (dWqkv, dWug, dWd, dWo)
    contract over the gathered tokens. By default they read the R row shards
    where they lie (fo_gemm_partials_sharded) and the all-gather GEMMs keep
    no gathered copy; `keep_gathered=True` has the all-gather GEMMs write the
    gathered inputs (Gx, Gh, G_dy, G_dh) and the weight gradients read those,
    as a framework that saves the gathered activation for its backward
    would."""

    def __init__(self, shape: LayerShape = LayerShape(), *, device="cuda", seed=4, mode="randn",
                 keep_gathered=False):
        self.s = s = shape
        R, T, H, F = s.R, s.T, s.H, s.F
        if T % R or H % R or F % R:
            raise ValueError("T, H and F must be divisible by R")
        dev = torch.device(device)
        g = torch.Generator().manual_seed(seed)
        w = (lambda shp: _ints(g, shp, dev)) if mode == "int" else (lambda shp: _draw(g, shp, 0.02, dev))
        a = (lambda shp: _ints(g, shp, dev)) if mode == "int" else (lambda shp: _draw(g, shp, 1.0, dev))
        bf, f32 = torch.bfloat16, torch.float32

        def per_rank(shp, dtype=bf):
            return [torch.empty(shp, dtype=dtype, device=dev) for _ in range(R)]

        def token_shards(draw, shp):
            # The R token shards of a sequence-parallel tensor, back to back
            # in rank order: their all-gather is the whole buffer.
            whole = torch.cat([draw(shp) for _ in range(R)]) if draw else torch.empty((R * shp[0], shp[1]),
                                                                                      dtype=bf, device=dev)
            return list(whole.split(shp[0]))

        # weights (each rank's slice)
        self.Wqkv = [w((H, 3 * H // R)) for _ in range(R)]
        self.Wo = [w((H // R, H)) for _ in range(R)]
        self.Wug = [w((H, 2 * F // R)) for _ in range(R)]
        self.Wd = [w((F // R, H)) for _ in range(R)]
        # forward inputs and the synthetic outputs of the skipped parts
        self.x = token_shards(a, (T // R, H))
        self.attn = [a((T, H // R)) for _ in range(R)]
        self.act = [a((T, F // R)) for _ in range(R)]
        # upstream gradients
        self.dy = token_shards(a, (T // R, H))              # into the down projection's output
        self.dh = token_shards(a, (T // R, H))              # into the o projection's output
        self.dug = [a((T, 2 * F // R)) for _ in range(R)]   # into up|gate's output (through SwiGLU)
        self.dqkv = [a((T, 3 * H // R)) for _ in range(R)]  # into QKV's output (through attention)
        # forward outputs (and, if kept, the gathered inputs for the weight gradients)
        self.keep_gathered = keep_gathered
        gathered = per_rank if keep_gathered else (lambda shp: None)
        self.Gx, self.Gh = gathered((T, H)), gathered((T, H))
        self.y_qkv, self.y_ug = per_rank((T, 3 * H // R)), per_rank((T, 2 * F // R))
        self.h, self.y = token_shards(None, (T // R, H)), per_rank((T // R, H))
        # backward outputs
        self.G_dy, self.G_dh = gathered((T, H)), gathered((T, H))
        self.d_act, self.d_attn = per_rank((T, F // R)), per_rank((T, H // R))
        self.d_h_from_ug, self.d_x = per_rank((T // R, H)), per_rank((T // R, H))
        self.dWd, self.dWo = per_rank((H, F // R), f32), per_rank((H, H // R), f32)   # [out x in]
        self.dWug, self.dWqkv = per_rank((H, 2 * F // R), f32), per_rank((H, 3 * H // R), f32)

        P = {}
        # forward
        P["qkv"] = B.fo_plan("ag_gemm", R, T, 3 * H, H)
        P["o"] = B.fo_plan("gemm_rs", R, T, H, H, out_dtype="bf16")
        P["ug"] = B.fo_plan("ag_gemm", R, T, 2 * F, H)
        P["down"] = B.fo_plan("gemm_rs", R, T, H, F, out_dtype="bf16")
        # backward: data gradients
        P["down_dx"] = B.fo_plan("ag_gemm", R, T, F, H, w_layout="nk")
        P["ug_dx"] = B.fo_plan("gemm_rs", R, T, H, 2 * F, w_layout="nk", out_dtype="bf16")
        P["o_dx"] = B.fo_plan("ag_gemm", R, T, H, H, w_layout="nk")
        P["qkv_dx"] = B.fo_plan("gemm_rs", R, T, H, 3 * H, w_layout="nk", out_dtype="bf16")
        # backward: weight gradients (per-rank GEMMs, no collective)
        P["down_dw"] = B.fo_plan("dp_grad_rs", R, H, F // R, T)
        P["ug_dw"] = B.fo_plan("dp_grad_rs", R, H, 2 * F // R, T)
        P["o_dw"] = B.fo_plan("dp_grad_rs", R, H, H // R, T)
        P["qkv_dw"] = B.fo_plan("dp_grad_rs", R, H, 3 * H // R, T)
        self.plans = P
        self.ws = {}
        for k, p in P.items():
            self.ws[k] = torch.empty(B.fo_workspace_size(p), dtype=torch.uint8, device=dev)
            B.fo_workspace_init(p, self.ws[k])
        self.launches = 0

    def forward(self, stream=None):
        P, ws = self.plans, self.ws
        B.fo_ag_gemm(P["qkv"], self.x, self.Wqkv, self.y_qkv, self.Gx, ws["qkv"], stream)
        B.fo_gemm_rs(P["o"], self.attn, self.Wo, self.h, ws["o"], stream)
        B.fo_ag_gemm(P["ug"], self.h, self.Wug, self.y_ug, self.Gh, ws["ug"], stream)
        B.fo_gemm_rs(P["down"], self.act, self.Wd, self.y, ws["down"], stream)
        self.launches += 4

    def _weight_grad(self, key, G, shards, dY, dW, stream):
        """dW_r = AllGather(shards)^T . dY_r for every rank: from the
        gathered copy G when it was kept, else from the shards in place."""
        if G is not None:
            B.fo_gemm_partials(self.plans[key], G, dY, dW, self.ws[key], stream)
        else:
            B.fo_gemm_partials_sharded(self.plans[key], shards, dY, dW, self.ws[key], stream)

    def backward(self, stream=None):
        P, ws = self.plans, self.ws
        # down (row-parallel): dAct = AG(dy) . Wd^T, dWd^T = AG(dy)^T . act
        B.fo_ag_gemm(P["down_dx"], self.dy, self.Wd, self.d_act, self.G_dy, ws["down_dx"], stream)
        self._weight_grad("down_dw", self.G_dy, self.dy, self.act, self.dWd, stream)
        # up|gate (column-parallel): dh = RS(dug . Wug^T), dWug = AG(h)^T . dug
        B.fo_gemm_rs(P["ug_dx"], self.dug, self.Wug, self.d_h_from_ug, ws["ug_dx"], stream)
        self._weight_grad("ug_dw", self.Gh, self.h, self.dug, self.dWug, stream)
        # o (row-parallel): dAttn = AG(dh) . Wo^T, dWo^T = AG(dh)^T . attn
        B.fo_ag_gemm(P["o_dx"], self.dh, self.Wo, self.d_attn, self.G_dh, ws["o_dx"], stream)
        self._weight_grad("o_dw", self.G_dh, self.dh, self.attn, self.dWo, stream)
        # QKV (column-parallel): dx = RS(dqkv . Wqkv^T), dWqkv = AG(x)^T . dqkv
        B.fo_gemm_rs(P["qkv_dx"], self.dqkv, self.Wqkv, self.d_x, ws["qkv_dx"], stream)
        self._weight_grad("qkv_dw", self.Gx, self.x, self.dqkv, self.dWqkv, stream)
        self.launches += 8

    def status(self) -> List[int]:
        return [B.fo_status_query(p, self.ws[k])[0] for k, p in self.plans.items()]
