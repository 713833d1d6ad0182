"""ctypes binding over the C ABI in include/moe.h (argument marshalling only).

Every stage runs in the CUDA library libmoe_gb300.so; this module checks
tensor devices / dtypes / shapes, allocates outputs with PyTorch, passes
`data_ptr()`s and the current CUDA stream, and turns a non-zero moe_status
into an exception. There is no fallback: if the library is missing, every
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

GATING = {"softmax_topk": 0, "softmax_all": 1}
ACT = {"swiglu": 0, "swiglu_oai": 1, "relu2": 2}
LAYOUT = {"packed": 0, "interleaved": 1}
SET_ALPHA, SET_BETA, SET_LIMIT = 1, 2, 4
FFN_KERNEL = {"auto": 0, "tiled": 1, "swap": 2}
ABI_VERSION = 4

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT",
          6: "MOE_ERR_MISALIGNED"}


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class MoeParams(ctypes.Structure):
    _fields_ = [("gating", ctypes.c_int32), ("activation", ctypes.c_int32),
                ("w13_layout", ctypes.c_int32), ("set", ctypes.c_uint32),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("limit", ctypes.c_float),
                ("ffn_kernel", ctypes.c_int32), ("expert_map", ctypes.c_void_p),
                ("n_local_experts", ctypes.c_int32)]


class RoutingMeta(ctypes.Structure):
    _fields_ = [("col_sum", ctypes.c_void_p), ("offs", ctypes.c_void_p),
                ("col_sorted", ctypes.c_void_p), ("row_sorted", ctypes.c_void_p),
                ("gate_scal", ctypes.c_void_p)]


_LIB = None

# name -> (restype, argtypes)
_P, _I64, _I32, _SZ, _U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t,
                             ctypes.c_uint64)
_PP = ctypes.POINTER(MoeParams)
_PM = ctypes.POINTER(RoutingMeta)
SIGNATURES = {
    "moe_abi_version": (_I32, []),
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_workspace_size": (_SZ, [_I64, _I32, _I32, _I32, _I32]),
    "moe_workspace_init": (_I32, [_P, _SZ, _P]),
    "moe_workspace_regions": (_I32, [_I64, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_route": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "moe_build_metadata": (_I32, [_P, _P, _I64, _I32, _I32, _PM, _P, _SZ, _P]),
    "moe_route_metadata": (_I32, [_P, _I64, _I32, _I32, _I32, _P, _P, _PM, _P, _SZ, _P]),
    "moe_build_metadata_noalloc": (_I32, [_P, _P, _I64, _I32, _I32, _PM, _P, _P]),
    "moe_grouped_ffn": (_I32, [_P, _PM, _P, _P, _I64, _I32, _I32, _I32, _I32, _PP, _P, _P, _SZ,
                               _P]),
    "moe_combine": (_I32, [_P, _I64, _I32, _I32, _P, _P]),
    "moe_forward": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _PP, _P, _P, _P, _PM,
                           _P, _SZ, _P]),
    "moe_forward_timed": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _PP, _P, _P, _P,
                                 _PM, _P, _SZ, _P, _I32, _P]),
    "moe_route_gemm": (_I32, [_P, _P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "moe_forward_gate": (_I32, [_P, _P, _P, _P, _I64, _I32, _I32, _I32, _I32, _PP, _P, _P, _P,
                                _PM, _P, _SZ, _P]),
    "moe_forward_launch_count": (_I32, [_I64, _I32, _I32, _I32, _I32]),
    "moe_ffn_plan": (_I32, [_I64, _I32, _I32, _I32, _I32, _P, _P]),
    "moe_read_status": (_I32, [_P, _SZ, _I32, _P]),
    "moe_selftest_wait_timeout": (_I32, [_P, _SZ, _U64, _P]),
}


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libmoe_gb300.so (built by `__graft_entry__.build()` or
    `python -m mixture_experts_routing_warp_gb300.build`). Raises if absent."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first "
                               "(python -m mixture_experts_routing_warp_gb300.build)")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        if L.moe_abi_version() != ABI_VERSION:
            raise RuntimeError("libmoe_gb300.so ABI version mismatch")
        _LIB = L
    return _LIB


def _check(status: int, what: str) -> None:
    if status != 0:
        raise MoEError(status, what)


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def make_params(gating: str = "softmax_topk", act: str = "swiglu", layout: str = "packed",
                alpha: Optional[float] = None, beta: Optional[float] = None,
                limit: Optional[float] = None, ffn_kernel: str = "auto",
                expert_map: Optional[torch.Tensor] = None,
                n_local_experts: Optional[int] = None) -> MoeParams:
    """moe_params with the `set` bits of the values that are not None, so
    unset parameters keep the activation's defaults. ffn_kernel picks the
    grouped-GEMM kernel: "auto", "tiled" (large per-expert batches) or
    "swap" (small ones). expert_map (int32 [E] on the device: local expert id
    or -1) and n_local_experts make moe_forward compute an expert-parallel
    rank's share; the params keep a reference to the map tensor."""
    p = MoeParams(GATING[gating], ACT[act], LAYOUT[layout], 0, 0.0, 0.0, 0.0,
                  FFN_KERNEL[ffn_kernel], None, 0)
    if expert_map is not None:
        _need(expert_map, "expert_map", torch.int32)
        if n_local_experts is None:
            raise ValueError("an expert map needs n_local_experts")
        p.expert_map = expert_map.data_ptr()
        p.n_local_experts = int(n_local_experts)
        p._map_tensor = expert_map
    if alpha is not None:
        p.set |= SET_ALPHA
        p.alpha = float(alpha)
    if beta is not None:
        p.set |= SET_BETA
        p.beta = float(beta)
    if limit is not None:
        p.set |= SET_LIMIT
        p.limit = float(limit)
    return p


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def workspace_size(n: int, E: int, k: int, H: int, I: int) -> int:
    return int(lib().moe_workspace_size(n, E, k, H, I))


WS_REGIONS = ("ctrl", "frows", "hist", "topk_indx", "topk_vals", "col_sum", "offs", "col_sorted",
              "row_sorted", "gate_scal", "sync", "sk_part", "x_sorted", "h", "y_flat")


def workspace_regions(n: int, E: int, k: int, H: int, I: int) -> dict:
    """name -> (byte offset, bytes used) of each workspace region."""
    off = (ctypes.c_size_t * len(WS_REGIONS))()
    used = (ctypes.c_size_t * len(WS_REGIONS))()
    _check(lib().moe_workspace_regions(n, E, k, H, I, off, used), "moe_workspace_regions")
    return {name: (int(off[i]), int(used[i])) for i, name in enumerate(WS_REGIONS)}


def workspace(n: int, E: int, k: int, H: int, I: int,
              device: Optional[torch.device] = None) -> torch.Tensor:
    """Allocate (with PyTorch) and initialise a workspace for these sizes."""
    size = workspace_size(n, E, k, H, I)
    if size == 0:
        raise ValueError("invalid sizes for moe_workspace_size")
    device = torch.device("cuda") if device is None else torch.device(device)
    ws = torch.empty(size, dtype=torch.uint8, device=device)
    _check(lib().moe_workspace_init(_ptr(ws), size, _stream(ws.device)), "moe_workspace_init")
    return ws


def route(logits: torch.Tensor, k: int, gating: str = "softmax_topk"):
    """Router top-k -> (topk_indx int32 [n, k], topk_vals bf16 [n, k])."""
    _need(logits, "logits", torch.float32)
    n, E = logits.shape
    indx = torch.empty((n, k), dtype=torch.int32, device=logits.device)
    vals = torch.empty((n, k), dtype=torch.bfloat16, device=logits.device)
    _check(lib().moe_route(_ptr(logits), n, E, k, GATING[gating], _ptr(indx), _ptr(vals),
                           _stream(logits.device)), "moe_route")
    return indx, vals


def empty_meta(N: int, E: int, device) -> dict:
    return {"col_sum": torch.empty(E, dtype=torch.int32, device=device),
            "offs": torch.empty(E + 1, dtype=torch.int32, device=device),
            "col_sorted": torch.empty(N, dtype=torch.int32, device=device),
            "row_sorted": torch.empty(N, dtype=torch.int32, device=device),
            "gate_scal": torch.empty(N, dtype=torch.bfloat16, device=device)}


def _meta_struct(m: dict) -> RoutingMeta:
    return RoutingMeta(m["col_sum"].data_ptr(), m["offs"].data_ptr(), m["col_sorted"].data_ptr(),
                       m["row_sorted"].data_ptr(), m["gate_scal"].data_ptr())


def build_metadata(topk_indx: torch.Tensor, topk_vals: torch.Tensor, E: int,
                   ws: torch.Tensor, meta: Optional[dict] = None) -> dict:
    """Routing metadata -> dict(col_sum, offs, col_sorted, row_sorted,
    gate_scal). gather = (col_sorted, row_sorted), scatter = (row_sorted, col_sorted)."""
    _need(topk_indx, "topk_indx", torch.int32)
    n, k = topk_indx.shape
    _need(topk_vals, "topk_vals", torch.bfloat16, (n, k))
    m = meta if meta is not None else empty_meta(n * k, E, topk_indx.device)
    _check(lib().moe_build_metadata(_ptr(topk_indx), _ptr(topk_vals), n, E, k,
                                    ctypes.byref(_meta_struct(m)), _ptr(ws), ws.numel(),
                                    _stream(topk_indx.device)), "moe_build_metadata")
    return m


def route_metadata(logits: torch.Tensor, k: int, E: Optional[int] = None,
                   gating: str = "softmax_topk", ws: Optional[torch.Tensor] = None,
                   meta: Optional[dict] = None, topk: Optional[tuple] = None):
    """Stages 1 + 2 in one call -> (topk_indx, topk_vals, meta dict)."""
    _need(logits, "logits", torch.float32)
    n, E = logits.shape
    if ws is None:
        ws = workspace(max(n, 1), E, k, 64, 64, logits.device)
    indx, vals = topk if topk is not None else (
        torch.empty((n, k), dtype=torch.int32, device=logits.device),
        torch.empty((n, k), dtype=torch.bfloat16, device=logits.device))
    m = meta if meta is not None else empty_meta(n * k, E, logits.device)
    _check(lib().moe_route_metadata(_ptr(logits), n, E, k, GATING[gating], _ptr(indx), _ptr(vals),
                                    ctypes.byref(_meta_struct(m)), _ptr(ws), ws.numel(),
                                    _stream(logits.device)), "moe_route_metadata")
    return indx, vals, m


def _intermediate(w13: torch.Tensor, params: MoeParams) -> int:
    """I from w13's rows: 2I for the gated activations, I for ReLU2."""
    rows = w13.shape[1]
    return rows if params.activation == ACT["relu2"] else rows // 2


def grouped_ffn(x: torch.Tensor, meta: dict, w13: torch.Tensor, w2: torch.Tensor, k: int,
                ws: torch.Tensor, params: MoeParams,
                y_flat: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gate-weighted per-expert FFN -> y_flat bf16 [n*k, H] in token-slot order."""
    _need(x, "x", torch.bfloat16)
    n, H = x.shape
    _need(w13, "w13", torch.bfloat16)
    E = w13.shape[0]
    I = _intermediate(w13, params)
    _need(w13, "w13", torch.bfloat16, (E, w13.shape[1], H))
    _need(w2, "w2", torch.bfloat16, (E, H, I))
    if y_flat is None:
        y_flat = torch.empty((n * k, H), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_grouped_ffn(_ptr(x), ctypes.byref(_meta_struct(meta)), _ptr(w13), _ptr(w2),
                                 n, E, k, H, I, ctypes.byref(params), _ptr(y_flat),
                                 _ptr(ws), ws.numel(), _stream(x.device)), "moe_grouped_ffn")
    return y_flat


def combine(y_flat: torch.Tensor, n: int, k: int,
            out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _need(y_flat, "y_flat", torch.bfloat16)
    H = y_flat.shape[1]
    if out is None:
        out = torch.empty((n, H), dtype=torch.bfloat16, device=y_flat.device)
    _check(lib().moe_combine(_ptr(y_flat), n, k, H, _ptr(out), _stream(y_flat.device)),
           "moe_combine")
    return out


def forward(x: torch.Tensor, logits: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor, k: int,
            params: MoeParams, ws: torch.Tensor, out: Optional[torch.Tensor] = None,
            topk: Optional[tuple] = None, meta: Optional[dict] = None) -> torch.Tensor:
    """The whole layer in one library call. `topk` = (indx, vals) and `meta`
    (dict of the five arrays) are optional outputs."""
    _need(x, "x", torch.bfloat16)
    n, H = x.shape
    _need(logits, "logits", torch.float32)
    E = logits.shape[1]
    E_w = params.n_local_experts if params.expert_map else E  # experts held in w13 / w2
    _need(w13, "w13", torch.bfloat16)
    I = _intermediate(w13, params)
    _need(w13, "w13", torch.bfloat16, (E_w, w13.shape[1], H))
    _need(w2, "w2", torch.bfloat16, (E_w, H, I))
    if out is None:
        out = torch.empty((n, H), dtype=torch.bfloat16, device=x.device)
    indx, vals = topk if topk is not None else (None, None)
    mstruct = ctypes.byref(_meta_struct(meta)) if meta is not None else None
    _check(lib().moe_forward(_ptr(x), _ptr(logits), _ptr(w13), _ptr(w2), n, E, k, H, I,
                             ctypes.byref(params), _ptr(out), _ptr(indx), _ptr(vals), mstruct,
                             _ptr(ws), ws.numel(), _stream(x.device)), "moe_forward")
    return out


def route_gemm(x: torch.Tensor, w_gate: torch.Tensor, k: int, gating: str = "softmax_topk",
               ws: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None):
    """Router matmul x . w_gate^T fused with the top-k -> (topk_indx, topk_vals);
    fills `logits` (fp32 [n, E]) too when given."""
    _need(x, "x", torch.bfloat16)
    n, H = x.shape
    _need(w_gate, "w_gate", torch.bfloat16)
    E = w_gate.shape[0]
    _need(w_gate, "w_gate", torch.bfloat16, (E, H))
    if logits is not None:
        _need(logits, "logits", torch.float32, (n, E))
    if ws is None:
        ws = workspace(max(n, 1), E, k, 64, 64, x.device)
    indx = torch.empty((n, k), dtype=torch.int32, device=x.device)
    vals = torch.empty((n, k), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_route_gemm(_ptr(x), _ptr(w_gate), n, E, H, k, GATING[gating], _ptr(indx),
                                _ptr(vals), _ptr(logits), _ptr(ws), ws.numel(),
                                _stream(x.device)), "moe_route_gemm")
    return indx, vals


def forward_gate(x: torch.Tensor, w_gate: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor,
                 k: int, params: MoeParams, ws: torch.Tensor, out: Optional[torch.Tensor] = None,
                 topk: Optional[tuple] = None, meta: Optional[dict] = None) -> torch.Tensor:
    """forward() with the routing computed from x and the gate weights [E, H]."""
    _need(x, "x", torch.bfloat16)
    n, H = x.shape
    _need(w_gate, "w_gate", torch.bfloat16)
    E = w_gate.shape[0]
    _need(w_gate, "w_gate", torch.bfloat16, (E, H))
    E_w = params.n_local_experts if params.expert_map else E  # experts held in w13 / w2
    _need(w13, "w13", torch.bfloat16)
    I = _intermediate(w13, params)
    _need(w13, "w13", torch.bfloat16, (E_w, w13.shape[1], H))
    _need(w2, "w2", torch.bfloat16, (E_w, H, I))
    if out is None:
        out = torch.empty((n, H), dtype=torch.bfloat16, device=x.device)
    indx, vals = topk if topk is not None else (None, None)
    mstruct = ctypes.byref(_meta_struct(meta)) if meta is not None else None
    _check(lib().moe_forward_gate(_ptr(x), _ptr(w_gate), _ptr(w13), _ptr(w2), n, E, k, H, I,
                                  ctypes.byref(params), _ptr(out), _ptr(indx), _ptr(vals),
                                  mstruct, _ptr(ws), ws.numel(), _stream(x.device)),
           "moe_forward_gate")
    return out


STAGES = ("route", "metadata", "gather", "ffn1", "ffn2", "combine")


def forward_timed(x: torch.Tensor, logits: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor,
                  k: int, params: MoeParams, ws: torch.Tensor, events: list,
                  out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """forward() that records len(STAGES) + 1 torch.cuda.Event objects between
    the stage kernels (events[i] before stage i, the last after the end)."""
    n, H = x.shape
    E = logits.shape[1]
    I = _intermediate(w13, params)
    if out is None:
        out = torch.empty((n, H), dtype=torch.bfloat16, device=x.device)
    if len(events) != len(STAGES) + 1:
        raise ValueError("need len(STAGES) + 1 events")
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().moe_forward_timed(_ptr(x), _ptr(logits), _ptr(w13), _ptr(w2), n, E, k, H, I,
                                   ctypes.byref(params), _ptr(out), None, None, None, _ptr(ws),
                                   ws.numel(), arr, len(events), _stream(x.device)),
           "moe_forward_timed")
    return out


def forward_launch_count(n: int, E: int, k: int, H: int, I: int) -> int:
    """Kernels one moe_forward enqueues for these sizes (-1: invalid sizes)."""
    return int(lib().moe_forward_launch_count(n, E, k, H, I))


def ffn_plan(n: int, E: int, k: int, H: int, I: int, params: MoeParams) -> dict:
    """How the two expert contractions are tiled for these sizes (no launch):
    token rows per tile of each, whether each runs on CTA pairs, whether the
    decode tiling applies, and whether both run in one launch."""
    plan = (ctypes.c_int32 * 6)()
    _check(lib().moe_ffn_plan(n, E, k, H, I, ctypes.byref(params), plan), "moe_ffn_plan")
    return {"token_tile_w13": plan[0], "token_tile_w2": plan[1], "pair_w13": bool(plan[2]),
            "pair_w2": bool(plan[3]), "decode": bool(plan[4]), "fused": bool(plan[5])}


def read_status(ws: torch.Tensor, reset: bool = False) -> int:
    """DEBUG: synchronises and returns the device status word (0 = OK)."""
    return int(lib().moe_read_status(_ptr(ws), ws.numel(), int(reset), _stream(ws.device)))


def selftest_wait_timeout(ws: torch.Tensor, timeout_ns: int) -> None:
    _check(lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel(), int(timeout_ns),
                                           _stream(ws.device)), "moe_selftest_wait_timeout")
