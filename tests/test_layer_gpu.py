"""The whole MoE layer on the GPU (through the C ABI) against the CPU oracle.

Routing and metadata must match bit for bit; the layer output within
|gpu - ref| <= 3e-2 + 2e-2 |ref| elementwise and cosine > 0.99.
Workloads: the tiny layer, the MiniMind layer (E = 4, 8, 16, top-1, softmax
over all experts), the GPT-OSS layer (decode n = 1, 8, 64 and prefill n = 2048 checked in
full; prefill n = 8192 on tokens from every 128-row block of every expert's
slice), the skewed 128-expert prefill (n = 16384, the same per-block tokens), and variants over layouts, activations,
activation parameters and ragged tile tails, each through both grouped-GEMM
kernels (tokens on the MMA's M side, and weights on it for small batches)."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import oracle
import moe_inputs as I

from helpers import assert_layer_close, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


class Layer:
    """Host inputs of a case plus their device copies and one GPU forward."""

    def __init__(self, case: I.LayerCase, act_kw=None, ffn_kernel: str = "auto"):
        self.case = case
        self.act_kw = act_kw or {}
        self.h = I.layer_inputs(case)
        self.x = dev_bf16(self.h["x"])
        self.logits = dev(self.h["logits"])
        self.w13 = dev_bf16(self.h["w13"])
        self.w2 = dev_bf16(self.h["w2"])
        self.params = moe.make_params(case.gating, case.act, case.layout, **self.act_kw,
                                      ffn_kernel=ffn_kernel)

    def forward(self):
        c = self.case
        ws = moe.workspace(c.n, c.E, c.k, c.H, c.I)
        indx = torch.empty((c.n, c.k), dtype=torch.int32, device="cuda")
        vals = torch.empty((c.n, c.k), dtype=torch.bfloat16, device="cuda")
        meta = moe.empty_meta(c.n * c.k, c.E, "cuda")
        out = moe.forward(self.x, self.logits, self.w13, self.w2, c.k, self.params, ws,
                          topk=(indx, vals), meta=meta)
        torch.cuda.synchronize()
        assert moe.read_status(ws) == 0
        return out, indx, vals, meta

    def oracle_kw(self):
        return dict(act=self.case.act, layout=self.case.layout, **self.act_kw)


def _check_routing(L, indx, vals, meta):
    ref_i, ref_v = oracle.route(L.h["logits"], L.case.k, L.case.gating)
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
    d = np.abs(host_bits(vals).astype(np.int32) - ref_v.astype(np.int32))
    assert d.max(initial=0) <= 1
    ref_m = oracle.metadata(indx.cpu().numpy(), host_bits(vals), L.case.E)
    for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
        np.testing.assert_array_equal(meta[key].cpu().numpy(), ref_m[key], err_msg=key)
    np.testing.assert_array_equal(host_bits(meta["gate_scal"]), ref_m["gate_scal"])
    return ref_m


def _check_full(L):
    out, indx, vals, meta = L.forward()
    _check_routing(L, indx, vals, meta)
    # the layer output is compared on the GPU's own routing (same bf16 gates)
    ref = oracle.ffn(L.h["x"], indx.cpu().numpy(), host_bits(vals), L.h["w13"], L.h["w2"],
                     **L.oracle_kw())
    return assert_layer_close(host_bits(out), ref, L.case.name)


def _tile_sample(meta: dict, k: int, rows: int = 128, seed: int = 123) -> np.ndarray:
    """Tokens covering every token tile of both contraction kernels: for each
    expert, one random sorted position in every 128-row block from the
    expert's first row (a CTA-pair half of a 256-row swap tile, a whole
    tiled-kernel tile) plus the expert's last row (its ragged tail)."""
    offs = meta["offs"].cpu().numpy()
    col_sorted = meta["col_sorted"].cpu().numpy()
    rng = np.random.default_rng(seed)
    pick = set()
    for e in range(offs.size - 1):
        a, b = int(offs[e]), int(offs[e + 1])
        for s0 in range(a, b, rows):
            pick.add(int(col_sorted[rng.integers(s0, min(s0 + rows, b))]) // k)
        if b > a:
            pick.add(int(col_sorted[b - 1]) // k)
    return np.array(sorted(pick), dtype=np.int64)


# oracle outputs already computed for a case's routing (both kernels share it)
_ORACLE_CACHE = {}


def _oracle_cached(L, indx: np.ndarray, vals_bits: np.ndarray, toks=None) -> np.ndarray:
    key = (L.case.name, indx.tobytes(), vals_bits.tobytes(),
           None if toks is None else toks.tobytes())
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()
        _ORACLE_CACHE[key] = oracle.ffn(L.h["x"], indx, vals_bits, L.h["w13"], L.h["w2"],
                                        tokens=toks, **L.oracle_kw())
    return _ORACLE_CACHE[key]


def _check_full_cached(L):
    """_check_full with the oracle's output reused across kernels."""
    out, indx, vals, meta = L.forward()
    _check_routing(L, indx, vals, meta)
    ref = _oracle_cached(L, indx.cpu().numpy(), host_bits(vals))
    return assert_layer_close(host_bits(out), ref, L.case.name)


def _check_tiles(L):
    """The layer on the tokens of _tile_sample (every token tile of every
    expert contributes rows), against the oracle."""
    out, indx, vals, meta = L.forward()
    _check_routing(L, indx, vals, meta)
    toks = _tile_sample(meta, L.case.k)
    ref = _oracle_cached(L, indx.cpu().numpy(), host_bits(vals), toks)
    return assert_layer_close(host_bits(out)[toks], ref, L.case.name)


def test_tiny_layer_and_golden():
    L = Layer(I.TINY)
    _check_full(L)
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "make_golden.py")
    spec = importlib.util.spec_from_file_location("make_golden", path)
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    g = mg.load()
    out, indx, _, meta = L.forward()
    np.testing.assert_array_equal(indx.cpu().numpy(), g["topk_indx"])
    for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
        np.testing.assert_array_equal(meta[key].cpu().numpy(), g[key])
    assert_layer_close(host_bits(out), g["out"], "tiny vs golden")


@pytest.mark.parametrize("case", [I.MINIMIND_E4, I.MINIMIND_E8, I.MINIMIND_E16],
                         ids=lambda c: c.name)
def test_minimind_layer(case):
    _check_full(Layer(case))


@pytest.mark.parametrize("n", I.GPTOSS_DECODE_N)
def test_gptoss_decode(n):
    L = Layer(I.GPTOSS.with_n(n))
    c = L.case
    plan = moe.ffn_plan(c.n, c.E, c.k, c.H, c.I, L.params)
    assert plan["decode"] == (c.n * c.k <= 32 * c.E)
    # both contractions in one launch at decode (and on pairs beyond it)
    assert plan["fused"] == (plan["decode"] or (plan["pair_w13"] and plan["pair_w2"]))
    _check_full(L)


@pytest.mark.parametrize("ffn_kernel", ["auto", "tiled"])
def test_gptoss_prefill_n2048_every_token(ffn_kernel):
    """GPT-OSS prefill at 2048 tokens: every output element against the oracle
    (AUTO: both contractions in one launch on CTA pairs)."""
    L = Layer(I.GPTOSS.with_n(2048), ffn_kernel=ffn_kernel)
    plan = moe.ffn_plan(2048, L.case.E, L.case.k, L.case.H, L.case.I, L.params)
    assert plan["fused"] == (ffn_kernel == "auto")
    _check_full_cached(L)


@pytest.mark.parametrize("ffn_kernel", ["auto", "tiled"])
def test_gptoss_prefill_n8192_every_tile(ffn_kernel):
    """GPT-OSS prefill at 8192 tokens: tokens from every 128-row block of
    every expert's slice (each CTA-pair half of each 256-row tile)."""
    L = Layer(I.GPTOSS.with_n(8192), ffn_kernel=ffn_kernel)
    plan = moe.ffn_plan(8192, L.case.E, L.case.k, L.case.H, L.case.I, L.params)
    if ffn_kernel == "auto":
        assert plan["pair_w13"] and plan["pair_w2"] and plan["fused"]
    _check_tiles(L)


@pytest.mark.parametrize("ffn_kernel", ["auto", "tiled"])
def test_skewed_prefill_every_tile(ffn_kernel):
    """The skewed 128-expert prefill (n = 16384; one expert holds almost every
    token, most hold 0-2): tokens from every 128-row block of every expert.
    AUTO runs both contractions in one launch on CTA pairs, where the w2
    tiles of the many tiny experts wait on few h rows each."""
    L = Layer(I.SKEWED, ffn_kernel=ffn_kernel)
    if ffn_kernel == "auto":
        c = L.case
        assert moe.ffn_plan(c.n, c.E, c.k, c.H, c.I, L.params)["fused"]
    _check_tiles(L)


VARIANTS = [
    # name, H, E, k, I, act, layout, act_kw
    ("packed_swiglu", 192, 8, 3, 320, "swiglu", "packed", {}),
    ("interleaved_swiglu", 192, 8, 3, 320, "swiglu", "interleaved", {}),
    ("packed_oai", 128, 6, 2, 192, "swiglu_oai", "packed", {}),
    ("interleaved_oai_params", 256, 5, 2, 128, "swiglu_oai", "interleaved",
     {"alpha": 1.5, "beta": 0.5, "limit": 3.0}),
    ("oai_limit_only", 128, 4, 4, 256, "swiglu_oai", "interleaved", {"limit": 2.0}),
    ("k8_e16", 64, 16, 8, 64, "swiglu", "packed", {}),
    # SiLU + clamp (a limit on plain SwiGLU) and the non-gated ReLU2
    ("silu_clamp_packed", 192, 8, 3, 320, "swiglu", "packed", {"limit": 0.5}),
    ("silu_clamp_interleaved", 128, 6, 2, 192, "swiglu", "interleaved", {"limit": 1.0}),
    ("relu2", 192, 8, 3, 320, "relu2", "packed", {}),
    ("relu2_k1", 256, 4, 1, 128, "relu2", "packed", {}),
]


@pytest.mark.parametrize("ffn_kernel", ["tiled", "swap"])
@pytest.mark.parametrize("name,H,E,k,Idim,act,layout,act_kw", VARIANTS,
                         ids=[v[0] for v in VARIANTS])
@pytest.mark.parametrize("n", [1, 37, 300])
def test_variants(name, H, E, k, Idim, act, layout, act_kw, n, ffn_kernel):
    case = I.LayerCase(f"{name}@n{n}", n=n, H=H, E=E, k=k, I=Idim, act=act, layout=layout,
                       seed=n, w_std=0.1)
    _check_full(Layer(case, act_kw, ffn_kernel))


def test_tiled_kernel_on_minimind():
    """The tiled kernel on 1024 rows per expert (8 token tiles each; the
    MiniMind test above runs the swap kernel's 256-row token tiles)."""
    _check_full(Layer(I.MINIMIND_E4, ffn_kernel="tiled"))


@pytest.mark.parametrize("n", I.GPTOSS_DECODE_N)
def test_gptoss_decode_tiled_kernel(n):
    """Decode through the tiled kernel too (AUTO picks the swap kernel there)."""
    _check_full(Layer(I.GPTOSS.with_n(n), ffn_kernel="tiled"))


@pytest.mark.parametrize("layout,act", [("packed", "swiglu"), ("interleaved", "swiglu_oai"),
                                        ("packed", "relu2")])
@pytest.mark.parametrize("n", [1, 5, 40, 300])
def test_swap_kernel_deep_k(layout, act, n):
    """The swap kernel with 16 K-blocks per tile in both contractions
    (H = I = 1024) and 1 .. 32 valid rows per tile (partial 8-column TMEM
    chunks); the result matches the oracle and repeats bit for bit."""
    case = I.LayerCase(f"deepk_{layout}@n{n}", n=n, H=1024, E=8, k=2, I=1024, act=act,
                       layout=layout, w_std=0.03, seed=n)
    L = Layer(case, ffn_kernel="swap")
    _check_full(L)
    c = case
    ws = moe.workspace(c.n, c.E, c.k, c.H, c.I)
    outs = [moe.forward(L.x, L.logits, L.w13, L.w2, c.k, L.params, ws).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_auto_kernel_choice_boundary():
    """n*k on both sides of 32*E: the swap kernel's token tiles switch from
    32 to 256 rows there; both widths correct."""
    for n in (64, 65):   # E = 8, k = 4: 256 = 32*8 -> swap, 260 -> tiled
        case = I.LayerCase(f"boundary@n{n}", n=n, H=128, E=8, k=4, I=192, w_std=0.1, seed=n)
        _check_full(Layer(case))


@pytest.mark.parametrize("act,layout", [("swiglu_oai", "interleaved"), ("relu2", "packed")])
def test_stages_compose_to_forward(act, layout):
    """route -> build_metadata -> grouped_ffn -> combine equals moe_forward bit for bit,
    and the per-slot outputs match the oracle's gate-weighted expert outputs."""
    case = I.LayerCase("stages", n=200, H=128, E=8, k=3, I=192, act=act, layout=layout,
                       w_std=0.1)
    L = Layer(case)
    out_fwd = L.forward()[0]
    ws = moe.workspace(case.n, case.E, case.k, case.H, case.I)
    indx, vals = moe.route(L.logits, case.k, case.gating)
    meta = moe.build_metadata(indx, vals, case.E, ws)
    y_flat = moe.grouped_ffn(L.x, meta, L.w13, L.w2, case.k, ws, L.params)
    out = moe.combine(y_flat, case.n, case.k)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_fwd.view(torch.int16))
    ref_out, y_slot, _ = oracle.ffn(L.h["x"], indx.cpu().numpy(), host_bits(vals), L.h["w13"],
                                    L.h["w2"], want_slots=True, **L.oracle_kw())
    ref_y = oracle.f64_to_bf16(y_slot.reshape(case.n * case.k, case.H))
    assert_layer_close(host_bits(y_flat), ref_y, "y_flat")
    assert_layer_close(host_bits(out), ref_out, "out")


@pytest.mark.parametrize("n,E,k,H,I_,act,layout", [
    (3, 32, 4, 256, 128, "swiglu_oai", "interleaved"),   # ~1 row per tile, stream-K w13
    (16, 32, 4, 256, 128, "swiglu", "packed"),           # n*k = 2 E
    (5, 5, 2, 128, 192, "swiglu_oai", "interleaved"),    # ragged groups of 4 rows
    (16, 8, 1, 128, 256, "relu2", "packed"),             # k = 1: w2 writes the output
])
def test_fused_gather_matches_materialised_rows(n, E, k, H, I_, act, layout):
    """With at most 2 slots per expert, moe_forward's w13 contraction fetches
    each tile's token rows from x (tile::gather4 of rows col_sorted[p] / k,
    only the tile's own rows); the stage path reads the rows the gather
    kernel materialised in X_sorted. Same arithmetic on the same rows: the
    outputs agree bit for bit. The forward launches no gather kernel there,
    and one kernel for both contractions."""
    assert moe.ffn_plan(n, E, k, H, I_, moe.make_params())["decode"]
    assert moe.forward_launch_count(n, E, k, H, I_) == 2 + (k > 1)
    case = I.LayerCase(f"fused_gather_n{n}", n=n, H=H, E=E, k=k, I=I_, act=act, layout=layout,
                       w_std=0.05, seed=n + E)
    L = Layer(case)
    out_fwd = L.forward()[0]
    ws = moe.workspace(case.n, case.E, case.k, case.H, case.I)
    indx, vals = moe.route(L.logits, case.k, case.gating)
    meta = moe.build_metadata(indx, vals, case.E, ws)
    y_flat = moe.grouped_ffn(L.x, meta, L.w13, L.w2, case.k, ws, L.params)
    out = y_flat if k == 1 else moe.combine(y_flat, case.n, case.k)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_fwd.view(torch.int16))
    _check_full(L)


@pytest.mark.parametrize("act,layout", [("swiglu_oai", "interleaved"), ("swiglu", "packed")])
def test_routing_kernel_rows_match_the_gather_kernel(act, layout):
    """With the cooperative route + metadata kernel on all SMs, moe_forward's
    dispatch rows are copied by that kernel after its scatter (no gather
    kernel); the stage path copies them with the gather kernel. Same rows,
    same arithmetic: the outputs agree bit for bit."""
    case = I.LayerCase(f"rows_in_routing_{act}", n=4096, H=256, E=32, k=4, I=128, act=act,
                       layout=layout, w_std=0.05, seed=41)
    # routing (with the rows), both contractions in one launch on CTA pairs, combine
    assert moe.forward_launch_count(case.n, case.E, case.k, case.H, case.I) == 3
    L = Layer(case)
    out_fwd = L.forward()[0]
    ws = moe.workspace(case.n, case.E, case.k, case.H, case.I)
    indx, vals = moe.route(L.logits, case.k, case.gating)
    meta = moe.build_metadata(indx, vals, case.E, ws)
    y_flat = moe.grouped_ffn(L.x, meta, L.w13, L.w2, case.k, ws, L.params)
    out = moe.combine(y_flat, case.n, case.k)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_fwd.view(torch.int16))


def test_empty_batch_is_a_noop():
    c = I.TINY
    L = Layer(c)
    ws = moe.workspace(0, c.E, c.k, c.H, c.I)
    x = torch.empty((0, c.H), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((0, c.E), dtype=torch.float32, device="cuda")
    out = moe.forward(x, logits, L.w13, L.w2, c.k, L.params, ws)
    torch.cuda.synchronize()
    assert out.shape == (0, c.H)


def _routed_case(counts, H=128, Idim=192, k=1, seed=0, act="swiglu", layout="packed"):
    """A layer whose top-1 routing sends exactly counts[e] tokens to expert e
    (the logits are built on the host so; the k-1 other slots go to the next
    experts in turn)."""
    E, n = len(counts), int(sum(counts))
    case = I.LayerCase(f"counts_{'_'.join(map(str, counts))}", n=n, H=H, E=E, k=k, I=Idim,
                       act=act, layout=layout, w_std=0.1, seed=seed)
    h = I.layer_inputs(case)
    owner = np.repeat(np.arange(E), counts)
    rng = np.random.default_rng(seed)
    owner = owner[rng.permutation(n)]
    logits = np.zeros((n, E), dtype=np.float32)
    for t in range(n):
        for j in range(k):
            logits[t, (owner[t] + j) % E] = float(k - j) + 1.0
    h["logits"] = logits
    return case, h


@pytest.mark.parametrize("ffn_kernel", ["auto", "tiled"])
@pytest.mark.parametrize("counts", [(256, 257, 32, 33), (128, 129, 1, 342), (0, 600, 0, 0)])
def test_tile_boundary_expert_loads(counts, ffn_kernel):
    """Experts holding exactly one, one-plus-one, or no token tile of either
    kernel (256 / 32 rows for the swap kernel, 128 for the tiled one)."""
    case, h = _routed_case(counts)
    L = Layer(case, ffn_kernel=ffn_kernel)
    L.h = h
    L.logits = dev(h["logits"])
    out, indx, vals, meta = L.forward()
    np.testing.assert_array_equal(meta["col_sum"].cpu().numpy(), np.array(counts))
    _check_routing(L, indx, vals, meta)
    ref = oracle.ffn(h["x"], indx.cpu().numpy(), host_bits(vals), h["w13"], h["w2"],
                     **L.oracle_kw())
    assert_layer_close(host_bits(out), ref, case.name)


@pytest.mark.parametrize("ffn_kernel", ["auto", "tiled"])
@pytest.mark.parametrize("E,k", [(1, 1), (4, 4), (8, 8)])
def test_degenerate_expert_counts(E, k, ffn_kernel):
    """E = 1 (a dense layer, gate weight 1) and k = E (every token to every
    expert)."""
    case = I.LayerCase(f"degenerate_e{E}_k{k}", n=130, H=128, E=E, k=k, I=128, w_std=0.1,
                       seed=E)
    _check_full(Layer(case, ffn_kernel=ffn_kernel))


@pytest.mark.parametrize("act,layout,Idim", [("swiglu_oai", "interleaved", 256),
                                             ("relu2", "packed", 512), ("swiglu", "packed", 256)])
def test_token_tile_widths(act, layout, Idim):
    """Sizes at which the swap kernel's width choice (least waves x per-tile
    cost) lands on 64-row token tiles for both contractions: n*k = 1200 rows
    over 8 experts with 4 weight tiles per expert on each side (32-row tiles
    would need two waves, 64-row ones fit one). The MiniMind tests cover the
    128-row choice."""
    case = I.LayerCase(f"ntw_{act}_{layout}", n=300, H=512, E=8, k=4, I=Idim, act=act,
                       layout=layout, w_std=0.05, seed=21)
    L = Layer(case)
    plan = moe.ffn_plan(case.n, case.E, case.k, case.H, case.I, L.params)
    assert (plan["token_tile_w13"], plan["token_tile_w2"]) == (64, 64)
    assert not (plan["pair_w13"] or plan["pair_w2"] or plan["decode"])
    _check_full(L)


@pytest.mark.parametrize("n,H,I_,act,layout", [
    (6144, 768, 768, "swiglu_oai", "interleaved"),   # one launch on CTA pairs
    (32, 256, 256, "swiglu", "packed"),              # decode (n*k <= 32E): stream-K units
])
def test_single_expert_in_one_launch(n, H, I_, act, layout):
    """E = 1 (a dense layer): in the launch that runs both contractions every
    w2 tile waits for all of the grid's w13 work. Against the oracle, twice,
    bit for bit."""
    case = I.LayerCase(f"one_expert_n{n}", n=n, H=H, E=1, k=1, I=I_, act=act, layout=layout,
                       w_std=0.05, seed=n)
    L = Layer(case)
    plan = moe.ffn_plan(n, 1, 1, H, I_, L.params)
    assert plan["fused"]
    _check_full(L)
    ws = moe.workspace(n, 1, 1, H, I_)
    outs = [moe.forward(L.x, L.logits, L.w13, L.w2, 1, L.params, ws).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("act,layout", [("swiglu_oai", "interleaved"), ("relu2", "packed"),
                                        ("swiglu", "packed")])
def test_cta_pair_tiles(act, layout):
    """Both contractions on CTA pairs (one M = 256 MMA over two SMs): 256-row
    token tiles in two waves. 384 weight rows per expert on each side, so the
    last pair tile's second CTA holds only rows past the end (zero-filled
    copies, skipped by the epilogue). The packed gated w13 reaches the kernel
    interleaved by its tensor map; there the past-the-end rows are gate/up
    pairs beyond I."""
    Idim = 384 if act == "relu2" else 192  # w13 rows: I or 2I = 384
    case = I.LayerCase(f"pairs_{act}", n=2048, H=384, E=8, k=4, I=Idim, act=act,
                       layout=layout, w_std=0.05, seed=31)
    L = Layer(case)
    plan = moe.ffn_plan(case.n, case.E, case.k, case.H, case.I, L.params)
    assert plan["token_tile_w13"] == 256 and plan["pair_w13"] and plan["pair_w2"]
    _check_full(L)


def test_cta_pair_ragged_expert_loads():
    """The pair MMA reads its first n_mma/2 token rows from the leader CTA and
    the rest from the peer: expert loads that leave last tiles of 1, 33, 164,
    20 and 255 rows move that split (16, 32, 96, 16, 128 rows)."""
    counts = (513, 1, 255, 257, 33, 0, 1700, 1300)
    case, h = _routed_case(counts, H=384, Idim=1536, act="swiglu_oai", layout="interleaved")
    L = Layer(case)
    L.h = h
    L.logits = dev(h["logits"])
    plan = moe.ffn_plan(case.n, case.E, case.k, case.H, case.I, L.params)
    assert plan["token_tile_w13"] == 256 and plan["pair_w13"]
    out, indx, vals, meta = L.forward()
    np.testing.assert_array_equal(meta["col_sum"].cpu().numpy(), np.array(counts))
    _check_routing(L, indx, vals, meta)
    ref = oracle.ffn(h["x"], indx.cpu().numpy(), host_bits(vals), h["w13"], h["w2"],
                     **L.oracle_kw())
    assert_layer_close(host_bits(out), ref, case.name)
