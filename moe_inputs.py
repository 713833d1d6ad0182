"""Seeded synthetic inputs for the MoE layer forward (test and benchmark
support, not part of the library package).

This module is the only code that both the CUDA path's tests/bench and the
CPU oracle's tests use. It draws random numbers and stores them as fp32 or
bf16; it holds none of the layer's arithmetic (no top-k, no softmax, no
sort, no FFN).

Every tensor comes from numpy's PCG64 (`np.random.default_rng`) keyed by a
tuple (seed, tensor tag, expert id), so that one expert's weights can be
regenerated alone (the oracle recomputes sampled tokens without building all
experts). Values are drawn in fp32 and stored as bf16 bit patterns (uint16)
with round-to-nearest-even.

Workload shapes follow the pages:
  * tiny layer: the parity-test shapes of the "Reuse topk SparseMatrix
    routing metadata in GPT-OSS MoE forward" report (section 关键源码片段,
    test_routing_data_from_sparse_topk_parity) scaled to a full layer;
  * MiniMind layer: hidden 512, 8x512 tokens, moe_intermediate 1408, top-1
    (issue "MoE feed-forward performs ~3xnum_experts device->host syncs per
    layer", section Measurement);
  * GPT-OSS layer: hidden 2880, 32 experts, top-4, intermediate 2880, w13
    interleaved [gate0, up0, gate1, ...] ("CuteDSL NVFP4 MoE adds SwiGLU-OAI
    and ReLU2" report, section 关键源码片段, reorder_w13_to_w31_for_flashinfer_cutedsl);
  * routing-only sweep: fp32 N(0,1) logits, n in {1, 33, 512, ...},
    (E, k) in {(32, 4), (128, 4)} (first report's parity test).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

# Tags that keep the random streams of different tensors apart.
_TAG_X, _TAG_WG, _TAG_W13, _TAG_W2, _TAG_LOGITS, _TAG_NOISE = 1, 2, 3, 4, 5, 6

GATING_TOPK = "softmax_topk"   # softmax over the k selected logits
GATING_ALL = "softmax_all"     # softmax over all E logits, keep the selected
ACT_SWIGLU = "swiglu"
ACT_SWIGLU_OAI = "swiglu_oai"
LAYOUT_PACKED = "packed"       # w13 rows [gate; up]
LAYOUT_INTERLEAVED = "interleaved"  # w13 rows [gate0, up0, gate1, up1, ...]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def normal_bf16(shape, std: float, *key: int) -> np.ndarray:
    """N(0, std^2) drawn in fp32 and stored as bf16 bits."""
    v = _rng(*key).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return f32_to_bf16_bits(v)


@dataclasses.dataclass(frozen=True)
class LayerCase:
    """One MoE layer workload: shapes, gating, activation, w13 layout, seed."""
    name: str
    n: int          # tokens
    H: int          # hidden
    E: int          # experts
    k: int          # experts per token (n_expts_act)
    I: int          # expert intermediate size
    gating: str = GATING_TOPK
    act: str = ACT_SWIGLU
    layout: str = LAYOUT_PACKED
    seed: int = 0
    router: str = "gemm"        # "gemm": logits = x W_g^T ; "skew": N(0,1) + b_e
    w_std: float = 0.02
    skew_scale: float = 2.0     # b_e = skew_scale * log(1 / (e+1)^skew_pow)
    skew_pow: float = 1.1

    def with_n(self, n: int) -> "LayerCase":
        return dataclasses.replace(self, n=n, name=f"{self.name.split('@')[0]}@n{n}")

    @property
    def flops(self) -> float:
        return 2.0 * self.n * self.k * self.H * 3 * self.I


# Workloads named by what they are.
TINY = LayerCase("tiny_n33_h64_e8_k2_i128", n=33, H=64, E=8, k=2, I=128)
MINIMIND_E4 = LayerCase("minimind_n4096_h512_e4_k1_i1408", n=4096, H=512, E=4, k=1,
                        I=1408, gating=GATING_ALL)
MINIMIND_E8 = dataclasses.replace(MINIMIND_E4, name="minimind_n4096_h512_e8_k1_i1408", E=8)
MINIMIND_E16 = dataclasses.replace(MINIMIND_E4, name="minimind_n4096_h512_e16_k1_i1408", E=16)
GPTOSS = LayerCase("gptoss_h2880_e32_k4_i2880", n=8192, H=2880, E=32, k=4, I=2880,
                   act=ACT_SWIGLU_OAI, layout=LAYOUT_INTERLEAVED)
SKEWED = LayerCase("skewed_n16384_h2880_e128_k4_i2880", n=16384, H=2880, E=128, k=4,
                   I=2880, act=ACT_SWIGLU_OAI, layout=LAYOUT_INTERLEAVED, router="skew")

ROUTE_SWEEP_N = (1, 33, 512, 4096, 16384)
ROUTE_SWEEP_EK = ((32, 4), (128, 4))
GPTOSS_DECODE_N = (1, 8, 64)
GPTOSS_PREFILL_N = (2048, 8192)


def route_logits(n: int, E: int, seed: int = 0, tie_heavy: bool = False) -> np.ndarray:
    """fp32 N(0,1) router logits [n, E].

    tie_heavy rounds them to bf16 (as the first report's test draws bf16
    logits), which makes exact ties between experts common."""
    v = _rng(seed, _TAG_LOGITS, n, E).standard_normal(size=(n, E), dtype=np.float32)
    if tie_heavy:
        v = bf16_bits_to_f32(f32_to_bf16_bits(v))
    return np.ascontiguousarray(v)


def small_int_logits(n: int, E: int, seed: int = 0, levels: int = 3) -> np.ndarray:
    """Logits drawn from a few integers: nearly every row holds ties."""
    v = _rng(seed, _TAG_LOGITS, n, E, levels).integers(-levels, levels + 1, size=(n, E))
    return np.ascontiguousarray(v.astype(np.float32))


def layer_x(case: LayerCase) -> np.ndarray:
    return normal_bf16((case.n, case.H), 1.0, case.seed, _TAG_X, case.n, case.H)


def router_weight(case: LayerCase) -> np.ndarray:
    return normal_bf16((case.E, case.H), case.w_std, case.seed, _TAG_WG, case.E, case.H)


def w13_rows(case: LayerCase) -> int:
    """Rows of one expert's w13: gate and up (2I), or w1 alone (I) for the
    non-gated ReLU2."""
    return case.I if case.act == "relu2" else 2 * case.I


def expert_w13(case: LayerCase, e: int) -> np.ndarray:
    """w13 of expert e, [2I, H] ([I, H] for ReLU2) bf16 bits, rows in the case's layout."""
    return normal_bf16((w13_rows(case), case.H), case.w_std, case.seed, _TAG_W13, e, case.I,
                       case.H)


def expert_w2(case: LayerCase, e: int) -> np.ndarray:
    """w2 of expert e, [H, I] bf16 bits."""
    return normal_bf16((case.H, case.I), case.w_std, case.seed, _TAG_W2, e, case.I, case.H)


def _per_expert(case: LayerCase, shape, fn) -> np.ndarray:
    """Stack fn(case, e) over experts; threads over experts (each expert has
    its own seed, so the result does not depend on the thread count)."""
    out = np.empty((case.E, *shape), dtype=np.uint16)

    def one(e):
        out[e] = fn(case, e)

    workers = max(1, min(case.E, os.cpu_count() or 1))
    if workers == 1 or out.nbytes < (8 << 20):
        for e in range(case.E):
            one(e)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(case.E)))
    return out


def all_w13(case: LayerCase) -> np.ndarray:
    return _per_expert(case, (w13_rows(case), case.H), expert_w13)


def all_w2(case: LayerCase) -> np.ndarray:
    return _per_expert(case, (case.H, case.I), expert_w2)


def layer_logits(case: LayerCase, x: Optional[np.ndarray] = None) -> np.ndarray:
    """fp32 router logits [n, E], computed once on the host.

    "gemm": logits = x W_g^T from the bf16 values, summed in float64 and
    stored as fp32 (the router matmul sits outside the layer path; both the
    oracle and the CUDA path receive these same logits).
    "skew": N(0,1) + b_e with b_e = skew_scale * log(1 / (e+1)^skew_pow),
    a Zipf-like load imbalance."""
    if case.router == "skew":
        noise = _rng(case.seed, _TAG_NOISE, case.n, case.E).standard_normal(
            size=(case.n, case.E), dtype=np.float32)
        e = np.arange(case.E, dtype=np.float64)
        bias = case.skew_scale * np.log(1.0 / np.power(e + 1.0, case.skew_pow))
        return np.ascontiguousarray((noise.astype(np.float64) + bias[None, :]).astype(np.float32))
    if x is None:
        x = layer_x(case)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    wg = bf16_bits_to_f32(router_weight(case)).astype(np.float64)
    return np.ascontiguousarray((xf @ wg.T).astype(np.float32))


def layer_inputs(case: LayerCase, weights: bool = True) -> dict:
    """All host inputs of one layer case: x, logits, and (optionally) w13, w2."""
    x = layer_x(case)
    d = {"x": x, "logits": layer_logits(case, x)}
    if weights:
        d["w13"] = all_w13(case)
        d["w2"] = all_w2(case)
    return d
