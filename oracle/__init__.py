"""CPU oracle for the MoE layer forward -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline /
reference leg may import this package. The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing from the
product: it is a separate, plain C implementation (`moe_oracle.c`, float64,
explicit loops and explicit stable orderings) plus this ctypes wrapper.

Functions, each following the pages (page title, section):
  route     -- top-k by logit (descending, ties to the lower expert id) and
               softmax gate weights; "Reuse topk SparseMatrix routing metadata
               in GPT-OSS MoE forward", 关键源码片段 (topk_fn(..., apply_softmax=True)),
               and the MiniMind issue, Summary (top-k weight of a softmax over all experts).
  metadata  -- col_sum, ragged offsets, col_sorted_indx / row_sorted_indx,
               gate_scal; first report, 关键源码片段 (routing_data_from_sparse_topk).
  ffn       -- per-expert SwiGLU / SwiGLU-OAI FFN and the gate-weighted
               combine (masked per-expert index_add_ formulation of the MiniMind
               issue, Summary; activations and w13 layouts of "CuteDSL NVFP4 MoE
               adds SwiGLU-OAI and ReLU2", 关键源码片段 and 评论区精华).
  forward   -- route -> metadata -> ffn.
  metadata and ffn take an optional expert map (expert parallelism: the
  rank's local id of each global expert, -1 for another rank's), under which
  slots of other ranks' experts are dropped; first report, 功能与动机 and
  风险与影响 (the -1 slots of an expert-parallel routing).

Pinning: `tests/test_oracle_*.py` check these against brute force on tiny
inputs, library routines (numpy stable argsort, bincount, argmax, float64
matmul), closed forms and invariants. `expert_row`'s pre-activation and the
whole-layer special cases are pinned; the absolute layer output for general
inputs rests on those pins (no worked example is printed on the pages).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import numpy as np

from . import build as _build

GATING = {"softmax_topk": 0, "softmax_all": 1}
ACT = {"swiglu": 0, "swiglu_oai": 1, "relu2": 2}
LAYOUT = {"packed": 0, "interleaved": 1}

# SwiGLU-OAI defaults ("CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2",
# 评论区精华: 1.702 / 1.0 / 7.0).
OAI_ALPHA, OAI_BETA, OAI_LIMIT = 1.702, 1.0, 7.0


class _ActParams(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int), ("layout", ctypes.c_int), ("alpha", ctypes.c_double),
                ("beta", ctypes.c_double), ("limit", ctypes.c_double)]


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int
        L.orc_route.argtypes = [p, i64, i32, i32, i32, p, p]
        L.orc_metadata.argtypes = [p, p, i64, i32, i32, p, i32, p, p, p, p, p]
        L.orc_expert_row.argtypes = [p, p, p, i32, i32, ctypes.POINTER(_ActParams), p, p, p]
        L.orc_ffn.argtypes = [p, p, p, p, p, i64, i32, i32, i32, i32, p, i32,
                              ctypes.POINTER(_ActParams), p, i64, p, p, p]
        L.orc_router_logits.argtypes = [p, p, i64, i32, i32, p]
        L.orc_router_logits.restype = ctypes.c_int
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16_array.argtypes = [p, i64, p]
        L.orc_num_threads.argtypes = []
        L.orc_num_threads.restype = ctypes.c_int
        for f in (L.orc_route, L.orc_metadata, L.orc_expert_row, L.orc_ffn):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def act_params(act: str = "swiglu", layout: str = "packed", alpha: Optional[float] = None,
               beta: Optional[float] = None, limit: Optional[float] = None) -> _ActParams:
    """Resolve activation parameters. Unset values take the activation's own
    defaults: SwiGLU-OAI 1.702 / 1.0 / 7.0; SwiGLU has no clamp unless a
    limit is given ("SILU + clamp"); ReLU2 takes no parameters."""
    if act == "swiglu_oai":
        a = OAI_ALPHA if alpha is None else alpha
        b = OAI_BETA if beta is None else beta
        lim = OAI_LIMIT if limit is None else limit
    elif act == "swiglu":
        a, b, lim = 1.0, 0.0, (math.inf if limit is None else limit)
    else:
        if limit is not None:
            raise ValueError("ReLU2 takes no clamp limit")
        a, b, lim = 1.0, 0.0, math.inf
    return _ActParams(ACT[act], LAYOUT[layout], float(a), float(b), float(lim))


def num_threads() -> int:
    """OpenMP threads the oracle's FFN runs with."""
    return int(lib().orc_num_threads())


def f64_to_bf16(v) -> np.ndarray:
    """float64 -> bf16 bits, one round-to-nearest-even step."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_f64_to_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def router_logits(x: np.ndarray, w_gate: np.ndarray, as_f32: bool = True) -> np.ndarray:
    """The router matmul: logits[t, e] = sum_h x[t, h] * w_gate[e, h] in float64
    (h ascending), rounded once to fp32 unless as_f32 is False.
    x [n, H], w_gate [E, H] bf16 bits."""
    x = _c(x, np.uint16)
    w = _c(w_gate, np.uint16)
    n, H = x.shape
    E, H2 = w.shape
    assert H2 == H
    out = np.empty((n, E), dtype=np.float64)
    _check(lib().orc_router_logits(_ptr(x), _ptr(w), n, E, H, _ptr(out)), "router_logits")
    return out.astype(np.float32) if as_f32 else out


def route(logits: np.ndarray, k: int, gating: str = "softmax_topk"):
    """-> topk_indx int32 [n, k], topk_vals bf16 bits [n, k]."""
    logits = _c(logits, np.float32)
    n, E = logits.shape
    indx = np.empty((n, k), dtype=np.int32)
    vals = np.empty((n, k), dtype=np.uint16)
    rc = lib().orc_route(_ptr(logits), n, E, k, GATING[gating], _ptr(indx), _ptr(vals))
    _check(rc, "route")
    return indx, vals


def _expert_map(expert_map, E: int, n_local: Optional[int]):
    if expert_map is None:
        return None, E
    m = _c(expert_map, np.int32)
    assert m.shape == (E,) and n_local is not None
    return m, int(n_local)


def metadata(topk_indx: np.ndarray, topk_vals: np.ndarray, E: int, expert_map=None,
             n_local: Optional[int] = None) -> dict:
    """-> dict(col_sum [E], offs [E+1], col_sorted [n*k], row_sorted [n*k],
    gate_scal [n*k] bf16 bits, gather_src, gather_dst, scatter_src, scatter_dst).

    expert_map [E] (expert parallelism): local id in [0, n_local) of each
    global expert, or -1 (expert on another rank). Then col_sum / offs cover
    the n_local local experts, col_sorted / gate_scal hold the offs[-1] kept
    slots, and row_sorted is -1 at dropped slots."""
    indx = _c(topk_indx, np.int32)
    vals = _c(topk_vals, np.uint16)
    n, k = indx.shape
    N = n * k
    emap, E_loc = _expert_map(expert_map, E, n_local)
    col_sum = np.empty(E_loc, dtype=np.int32)
    offs = np.empty(E_loc + 1, dtype=np.int32)
    col_sorted = np.empty(N, dtype=np.int32)
    row_sorted = np.empty(N, dtype=np.int32)
    gate_scal = np.empty(N, dtype=np.uint16)
    rc = lib().orc_metadata(_ptr(indx), _ptr(vals), n, E, k, _ptr(emap), E_loc, _ptr(col_sum),
                            _ptr(offs), _ptr(col_sorted), _ptr(row_sorted), _ptr(gate_scal))
    _check(rc, "metadata")
    kept = int(offs[-1])
    col_sorted, gate_scal = col_sorted[:kept], gate_scal[:kept]
    return {"col_sum": col_sum, "offs": offs, "col_sorted": col_sorted,
            "row_sorted": row_sorted, "gate_scal": gate_scal,
            # GatherIndx(src=combine_indx, dst=dispatch_indx),
            # ScatterIndx(src=dispatch_indx, dst=combine_indx)
            "gather_src": col_sorted, "gather_dst": row_sorted,
            "scatter_src": row_sorted, "scatter_dst": col_sorted}


def expert_row(x_row: np.ndarray, w13_e: np.ndarray, w2_e: np.ndarray, **act_kw):
    """One expert on one row -> (a float64 [rows], h bf16 bits [I], y float64 [H]);
    rows = 2I for the gated activations, I for ReLU2."""
    x_row = _c(x_row, np.uint16)
    w13_e = _c(w13_e, np.uint16)
    w2_e = _c(w2_e, np.uint16)
    rows, H = w13_e.shape
    I = rows if act_kw.get("act") == "relu2" else rows // 2
    assert w2_e.shape == (H, I) and x_row.shape == (H,)
    a = np.empty(rows, dtype=np.float64)
    h = np.empty(I, dtype=np.uint16)
    y = np.empty(H, dtype=np.float64)
    prm = act_params(**act_kw)
    rc = lib().orc_expert_row(_ptr(x_row), _ptr(w13_e), _ptr(w2_e), H, I, ctypes.byref(prm),
                              _ptr(a), _ptr(h), _ptr(y))
    _check(rc, "expert_row")
    return a, h, y


def ffn(x: np.ndarray, topk_indx: np.ndarray, topk_vals: np.ndarray, w13: np.ndarray,
        w2: np.ndarray, tokens: Optional[np.ndarray] = None, want_slots: bool = False,
        expert_map=None, n_experts: Optional[int] = None, **act_kw):
    """Gate-weighted per-expert FFN + combine.

    x [n, H] bf16 bits; w13 [E, 2I, H] (ReLU2: [E, I, H]), w2 [E, H, I] bf16 bits.
    tokens: optional token ids to compute (rows of the result follow it).
    expert_map [n_experts] (expert parallelism): w13 / w2 then hold the local
    experts, slot j uses local expert expert_map[topk_indx[t, j]], and slots
    mapped to -1 add nothing (zero y_slot / h_slot entries).
    Returns out bf16 bits [n_sel, H]; with want_slots also
    y_slot float64 [n_sel, k, H] (gate-weighted, slot order) and
    h_slot bf16 bits [n_sel, k, I]."""
    x = _c(x, np.uint16)
    indx = _c(topk_indx, np.int32)
    vals = _c(topk_vals, np.uint16)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    n, H = x.shape
    E_loc, rows, H2 = w13.shape
    I = rows if act_kw.get("act") == "relu2" else rows // 2
    k = indx.shape[1]
    assert H2 == H and w2.shape == (E_loc, H, I) and indx.shape == (n, k) == vals.shape
    E = E_loc if expert_map is None else int(n_experts)
    emap, E_loc = _expert_map(expert_map, E, E_loc)
    toks = None if tokens is None else _c(tokens, np.int64)
    n_sel = n if toks is None else toks.size
    out = np.empty((n_sel, H), dtype=np.uint16)
    y_slot = np.empty((n_sel, k, H), dtype=np.float64) if want_slots else None
    h_slot = np.empty((n_sel, k, I), dtype=np.uint16) if want_slots else None
    prm = act_params(**act_kw)
    rc = lib().orc_ffn(_ptr(x), _ptr(indx), _ptr(vals), _ptr(w13), _ptr(w2), n, E, k, H, I,
                       _ptr(emap), E_loc, ctypes.byref(prm), _ptr(toks), n_sel, _ptr(out),
                       _ptr(y_slot), _ptr(h_slot))
    _check(rc, "ffn")
    if want_slots:
        return out, y_slot, h_slot
    return out


def forward(x, logits, w13, w2, k: int, gating: str = "softmax_topk", tokens=None, **act_kw):
    """route -> metadata -> ffn; returns a dict of every stage's outputs."""
    E = w13.shape[0]
    indx, vals = route(logits, k, gating)
    meta = metadata(indx, vals, E)
    out = ffn(x, indx, vals, w13, w2, tokens=tokens, **act_kw)
    return {"topk_indx": indx, "topk_vals": vals, **meta, "out": out}
