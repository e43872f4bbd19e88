"""Thin ctypes binding of libflashoverlap.so (include/flashoverlap.h).

Argument marshalling only: device pointers and streams are taken from torch
tensors / streams, every step of the computation runs in the library's CUDA
kernels. Function names match the C ABI. A non-OK status raises
``FlashOverlapError``. If the library has not been built the first call
raises: there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_int32, c_int64, c_size_t, c_uint64, c_void_p
from typing import List, Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libflashoverlap.so")

FO_OK, FO_ERR_INVALID_ARG, FO_ERR_SHAPE, FO_ERR_DTYPE, FO_ERR_ALIGN = 0, 1, 2, 3, 4
FO_ERR_UNSUPPORTED, FO_ERR_CUDA, FO_ERR_TIMEOUT, FO_ERR_PLAN_INVARIANT = 5, 6, 7, 8
FO_ERR_SCRATCH_LIMIT = 9
FO_NOALLOC_SCRATCH_BYTES = 64 * 1024
OPS = {"ag_gemm": 0, "gemm_rs": 1, "dp_grad_rs": 2, "gemm_ar": 3, "gemm_a2a": 4}
DTYPES = {"bf16": 0, "f32": 1}
SCHEDS = {"rank_adaptive": 0, "sliced": 1}
TRANSPORTS = {"peer_read": 0, "copy": 1}
W_LAYOUTS = {"kn": 0, "nk": 1}
INJECT = {"none": 0, "drop_transfer": 1, "skip_signal": 2, "delay_first_task": 3}
FO_TRACE_STAMPS = 8
FO_TRACE_MAX_CTAS = 1024
TILE_CONFIGS = {"auto": 0, "single": 1}
INTERLEAVES = {"auto": 0, "lockstep": 1, "skewed": 2, "rank_major": 3, "skewed_pairs": 4}
RS_ALGOS = {"direct": 0, "ring": 1}
TAIL_SPLITS = {"auto": 0, "off": 1, "on": 2}

# Every symbol include/flashoverlap.h declares.
EXPORTED = [
    "fo_plan", "fo_plan_destroy", "fo_plan_table", "fo_plan_transfers", "fo_plan_edges",
    "fo_workspace_size", "fo_workspace_init", "fo_ag_gemm", "fo_gemm_rs", "fo_dp_grad_rs",
    "fo_status_query", "fo_gemm_partials", "fo_reduce_scatter_f32", "fo_all_gather_copy",
    "fo_plan_last_launches", "fo_status_string", "fo_version", "fo_gemm_rs_noalloc", "fo_plan_task_order",
    "fo_gemm_ar", "fo_trace_query", "fo_plan_last_split_tiles", "fo_check_device_pointers",
    "fo_gemm_a2a", "fo_all_to_all_copy", "fo_attn_rs", "fo_attention", "fo_gemm_partials_sharded",
]


class FlashOverlapError(RuntimeError):
    def __init__(self, code: int, where: str, info=None):
        self.code = code
        self.info = info
        msg = f"{where}: {status_string(code)} (code {code})"
        if info is not None:
            msg += f" info={list(info)}"
        super().__init__(msg)


class PlanDesc(ctypes.Structure):
    _fields_ = [
        ("op", c_int32), ("R", c_int32), ("M", c_int64), ("N", c_int64), ("K", c_int64),
        ("in_dtype", c_int32), ("out_dtype", c_int32), ("sched", c_int32), ("ag_transport", c_int32),
        ("w_layout", c_int32), ("deterministic", c_int32), ("timeout_ns", c_uint64),
        ("fault_inject", c_int32), ("tile_config", c_int32), ("interleave", c_int32), ("rs_algo", c_int32),
        ("trace", c_int32), ("inject_delay_us", c_int32), ("tail_split", c_int32),
        ("reserved", c_int32 * 1),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libflashoverlap.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libflashoverlap.so not found at {path}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P = c_void_p
    PP = POINTER(c_void_p)
    sig = {
        "fo_plan": ([POINTER(PlanDesc), POINTER(c_void_p)], c_int32),
        "fo_plan_destroy": ([P], None),
        "fo_plan_table": ([P, POINTER(c_int32)], c_int32),
        "fo_plan_task_order": ([P, POINTER(c_int32)], c_int32),
        "fo_plan_transfers": ([P, POINTER(c_int32), c_int32, POINTER(c_int32)], c_int32),
        "fo_plan_edges": ([P, POINTER(c_int32), c_int32, POINTER(c_int32)], c_int32),
        "fo_workspace_size": ([P, POINTER(c_size_t)], c_int32),
        "fo_workspace_init": ([P, P, P], c_int32),
        "fo_ag_gemm": ([P, PP, PP, PP, PP, P, P], c_int32),
        "fo_gemm_rs": ([P, PP, PP, PP, P, P], c_int32),
        "fo_dp_grad_rs": ([P, PP, PP, PP, P, P], c_int32),
        "fo_gemm_rs_noalloc": ([P, PP, PP, PP, P], c_int32),
        "fo_gemm_ar": ([P, PP, PP, PP, P, P], c_int32),
        "fo_gemm_a2a": ([P, PP, PP, PP, P, P], c_int32),
        "fo_all_to_all_copy": ([P, PP, PP, P], c_int32),
        "fo_attn_rs": ([P, PP, PP, PP, PP, PP, PP, c_int32, c_int32, P, P], c_int32),
        "fo_attention": ([P, PP, PP, PP, PP, c_int32, c_int32, P, P], c_int32),
        "fo_gemm_partials_sharded": ([P, PP, PP, PP, P, P], c_int32),
        "fo_status_query": ([P, P, P, POINTER(c_int32)], c_int32),
        "fo_trace_query": ([P, P, P, POINTER(ctypes.c_uint64), c_int32, POINTER(c_int32)], c_int32),
        "fo_gemm_partials": ([P, PP, PP, PP, P, P], c_int32),
        "fo_reduce_scatter_f32": ([P, PP, PP, P], c_int32),
        "fo_all_gather_copy": ([P, PP, PP, P], c_int32),
        "fo_plan_last_launches": ([P], c_int32),
        "fo_plan_last_split_tiles": ([P], c_int32),
        "fo_check_device_pointers": ([c_int32, PP, P], c_int32),
        "fo_status_string": ([c_int32], ctypes.c_char_p),
        "fo_version": ([], c_int32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().fo_status_string(code).decode()
    except Exception:  # library missing: still give a readable message
        return f"status {code}"


def _check(code: int, where: str):
    if code != FO_OK:
        raise FlashOverlapError(code, where)


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_contiguous():
            raise ValueError("tensors passed to libflashoverlap must be contiguous")
        if not getattr(x, "is_cuda", True) and not x.is_pinned():
            raise ValueError("tensors passed to libflashoverlap must be CUDA tensors (or pinned host memory)")
        return x.data_ptr()
    raise TypeError(f"cannot take a device pointer from {type(x)!r}")


def _ptr_array(xs: Optional[Sequence]):
    if xs is None:
        return None
    arr = (c_void_p * len(xs))()
    for i, x in enumerate(xs):
        arr[i] = _ptr(x)
    return arr


def _stream(s) -> int:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Plan:
    """Owns an fo_plan_t; freed with fo_plan_destroy when collected."""

    def __init__(self, handle: int, desc: PlanDesc):
        self.handle = handle
        self.desc = desc
        self.R = desc.R

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.fo_plan_destroy(self.handle)
            self.handle = None

    @property
    def _as_parameter_(self):
        return c_void_p(self.handle)


def fo_plan(op: str, R: int, M: int, N: int, K: int, *, in_dtype="bf16", out_dtype=None,
            sched="rank_adaptive", ag_transport="peer_read", w_layout="kn", deterministic=False,
            timeout_ns=0, fault_inject="none", tile_config="auto", interleave="auto",
            rs_algo="direct", trace=False, inject_delay_us=0, tail_split="auto") -> Plan:
    lib = load()
    if out_dtype is None:
        out_dtype = "bf16" if op in ("ag_gemm", "gemm_a2a") else "f32"
    d = PlanDesc()
    d.op = OPS[op]
    d.R = R
    d.M, d.N, d.K = M, N, K
    d.in_dtype = DTYPES[in_dtype]
    d.out_dtype = DTYPES[out_dtype]
    d.sched = SCHEDS[sched]
    d.ag_transport = TRANSPORTS[ag_transport]
    d.w_layout = W_LAYOUTS[w_layout]
    d.deterministic = 1 if deterministic else 0
    d.timeout_ns = timeout_ns
    d.fault_inject = INJECT[fault_inject]
    d.tile_config = TILE_CONFIGS[tile_config]
    d.interleave = INTERLEAVES[interleave]
    d.rs_algo = RS_ALGOS[rs_algo]
    d.trace = 1 if trace else 0
    d.inject_delay_us = inject_delay_us
    d.tail_split = TAIL_SPLITS[tail_split]
    h = c_void_p()
    _check(lib.fo_plan(ctypes.byref(d), ctypes.byref(h)), "fo_plan")
    return Plan(h.value, d)


def fo_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        load().fo_plan_destroy(plan.handle)
        plan.handle = None


def fo_plan_table(plan: Plan) -> List[List[int]]:
    R = plan.R
    buf = (c_int32 * (R * R))()
    _check(load().fo_plan_table(plan, buf), "fo_plan_table")
    return [[buf[r * R + s] for s in range(R)] for r in range(R)]


def fo_plan_task_order(plan: Plan):
    """[(rank, step), ...] in the order the kernel runs the chunk tasks."""
    n = plan.R * plan.R
    buf = (c_int32 * (2 * n))()
    _check(load().fo_plan_task_order(plan, buf), "fo_plan_task_order")
    return [(buf[2 * i], buf[2 * i + 1]) for i in range(n)]


def _quads(fn, plan: Plan, what: str):
    n = c_int32()
    fn(plan, None, 0, ctypes.byref(n))
    cap = max(n.value, 1)
    buf = (c_int32 * (4 * cap))()
    _check(fn(plan, buf, cap, ctypes.byref(n)), what)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n.value)]


def fo_plan_transfers(plan: Plan):
    return _quads(load().fo_plan_transfers, plan, "fo_plan_transfers")


def fo_plan_edges(plan: Plan):
    return _quads(load().fo_plan_edges, plan, "fo_plan_edges")


def fo_workspace_size(plan: Plan) -> int:
    n = c_size_t()
    _check(load().fo_workspace_size(plan, ctypes.byref(n)), "fo_workspace_size")
    return n.value


def fo_workspace_init(plan: Plan, ws, stream=None) -> None:
    _check(load().fo_workspace_init(plan, _ptr(ws), _stream(stream)), "fo_workspace_init")


def fo_gemm_rs(plan: Plan, X, W, Y, ws, stream=None) -> None:
    _check(load().fo_gemm_rs(plan, _ptr_array(X), _ptr_array(W), _ptr_array(Y), _ptr(ws), _stream(stream)),
           "fo_gemm_rs")


def fo_gemm_ar(plan: Plan, X, W, Y, ws, stream=None) -> None:
    _check(load().fo_gemm_ar(plan, _ptr_array(X), _ptr_array(W), _ptr_array(Y), _ptr(ws), _stream(stream)),
           "fo_gemm_ar")


def fo_gemm_a2a(plan: Plan, X, W, Y, ws, stream=None) -> None:
    _check(load().fo_gemm_a2a(plan, _ptr_array(X), _ptr_array(W), _ptr_array(Y), _ptr(ws), _stream(stream)),
           "fo_gemm_a2a")


def fo_all_to_all_copy(plan: Plan, P, Y, stream=None) -> None:
    _check(load().fo_all_to_all_copy(plan, _ptr_array(P), _ptr_array(Y), _stream(stream)), "fo_all_to_all_copy")


def fo_attn_rs(plan: Plan, Q, K, V, Wo, O, Y, heads: int, causal: bool, ws, stream=None) -> None:
    _check(load().fo_attn_rs(plan, _ptr_array(Q), _ptr_array(K), _ptr_array(V), _ptr_array(Wo), _ptr_array(O),
                             _ptr_array(Y), int(heads), 1 if causal else 0, _ptr(ws), _stream(stream)),
           "fo_attn_rs")


def fo_attention(plan: Plan, Q, K, V, O, heads: int, causal: bool, ws, stream=None) -> None:
    _check(load().fo_attention(plan, _ptr_array(Q), _ptr_array(K), _ptr_array(V), _ptr_array(O), int(heads),
                               1 if causal else 0, _ptr(ws), _stream(stream)),
           "fo_attention")


def fo_ag_gemm(plan: Plan, X, W, Y, G=None, ws=None, stream=None) -> None:
    _check(load().fo_ag_gemm(plan, _ptr_array(X), _ptr_array(W), _ptr_array(Y), _ptr_array(G), _ptr(ws),
                             _stream(stream)), "fo_ag_gemm")


def fo_gemm_rs_noalloc(plan: Plan, X, W, Y, stream=None) -> None:
    """fo_gemm_rs without a workspace (static device scratch; see the header)."""
    _check(load().fo_gemm_rs_noalloc(plan, _ptr_array(X), _ptr_array(W), _ptr_array(Y), _stream(stream)),
           "fo_gemm_rs_noalloc")


def fo_dp_grad_rs(plan: Plan, X, dY, dW, ws, stream=None) -> None:
    _check(load().fo_dp_grad_rs(plan, _ptr_array(X), _ptr_array(dY), _ptr_array(dW), _ptr(ws),
                                _stream(stream)), "fo_dp_grad_rs")


def fo_gemm_partials(plan: Plan, A, B, P, ws, stream=None) -> None:
    _check(load().fo_gemm_partials(plan, _ptr_array(A), _ptr_array(B), _ptr_array(P), _ptr(ws),
                                   _stream(stream)), "fo_gemm_partials")


def fo_gemm_partials_sharded(plan: Plan, A_shards, B, P, ws, stream=None) -> None:
    _check(load().fo_gemm_partials_sharded(plan, _ptr_array(A_shards), _ptr_array(B), _ptr_array(P), _ptr(ws),
                                           _stream(stream)), "fo_gemm_partials_sharded")


def fo_check_device_pointers(ptrs, stream=None) -> int:
    """Status of fo_check_device_pointers for raw addresses (ints): FO_OK
    when the current device can use every one of them."""
    arr = (c_void_p * len(ptrs))(*[int(p) for p in ptrs])
    return int(load().fo_check_device_pointers(len(ptrs), arr, _stream(stream)))


def fo_reduce_scatter_f32(plan: Plan, P, Y, stream=None) -> None:
    _check(load().fo_reduce_scatter_f32(plan, _ptr_array(P), _ptr_array(Y), _stream(stream)),
           "fo_reduce_scatter_f32")


def fo_all_gather_copy(plan: Plan, X, G, stream=None) -> None:
    _check(load().fo_all_gather_copy(plan, _ptr_array(X), _ptr_array(G), _stream(stream)), "fo_all_gather_copy")


def fo_status_query(plan: Plan, ws, stream=None):
    """Returns (status code, [code, rank, step, chunk]) without raising."""
    info = (c_int32 * 4)()
    code = load().fo_status_query(plan, _ptr(ws), _stream(stream), info)
    return code, list(info)


def fo_trace_query(plan: Plan, ws, stream=None):
    """Per-CTA timestamps of the last traced launch: a list with one row of
    FO_TRACE_STAMPS ints (ns) per CTA."""
    cap = FO_TRACE_MAX_CTAS
    buf = (ctypes.c_uint64 * (cap * FO_TRACE_STAMPS))()
    n = c_int32()
    _check(load().fo_trace_query(plan, _ptr(ws), _stream(stream), buf, cap, ctypes.byref(n)), "fo_trace_query")
    m = min(n.value, cap)
    return [[buf[i * FO_TRACE_STAMPS + j] for j in range(FO_TRACE_STAMPS)] for i in range(m)]


def trace_summary(stamps):
    """Launch span, end of the math and exposed tail (all ns) from
    fo_trace_query's rows: the tail is the time the last transfer was still
    running after the last MMA had completed."""
    start = min(r[0] for r in stamps)
    mma_end = max(r[1] for r in stamps)
    xfer_end = max(max(r[2:6]) for r in stamps)
    end = max(r[6] for r in stamps)
    return {"span_ns": end - start, "mma_end_ns": mma_end - start, "transfers_end_ns": xfer_end - start,
            "exposed_tail_ns": max(0, xfer_end - mma_end)}


def fo_plan_last_launches(plan: Plan) -> int:
    return load().fo_plan_last_launches(plan)


def fo_plan_last_split_tiles(plan: Plan) -> int:
    return load().fo_plan_last_split_tiles(plan)


def fo_version() -> int:
    return load().fo_version()
