"""moe_forward with an expert map (an expert-parallel rank's share of the
layer) on the GPU, through the C ABI, against the oracle's expert map.

"Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward",
功能与动机 (expert-parallel routing) and 风险与影响 (the -1 slots): the rank
holds a subset of the experts; top-k runs over all experts, slots of other
ranks' experts are dropped from the dispatch and add nothing to the output.
Routing (global ids) and the local metadata match bit for bit; the output
within the layer tolerance; tokens with no local slot get exact zero rows.
Covers the one-CTA decode kernel, the fused gather, the cooperative route +
metadata kernel over many CTAs, k = 1 (which then goes through the
combine), the router matmul path and permuted local ids."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import oracle
import moe_inputs as I

from helpers import assert_layer_close, dev, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def _rank_map(E, ranks, r, permute=False):
    m = np.full(E, -1, dtype=np.int32)
    mine = np.arange(E)[np.arange(E) * ranks // E == r]
    loc = np.arange(mine.size)
    if permute:
        loc = np.random.default_rng(E + r).permutation(mine.size)
    m[mine] = loc
    inv = np.empty(mine.size, dtype=np.int64)
    inv[loc] = mine  # local id -> global expert
    return m, inv


def _run(case, m, inv, gate=False, ffn_kernel="auto"):
    h = I.layer_inputs(case)
    if gate:  # routing from the router matmul: the oracle routes the GPU's logits
        w_gate = I.router_weight(case)
    n, E, k = case.n, case.E, case.k
    E_loc = inv.size
    emap = dev(m)
    params = moe.make_params(case.gating, case.act, case.layout, expert_map=emap,
                             n_local_experts=E_loc, ffn_kernel=ffn_kernel)
    x = dev_bf16(h["x"])
    w13 = dev_bf16(h["w13"][inv])
    w2 = dev_bf16(h["w2"][inv])
    ws = moe.workspace(n, E, k, case.H, case.I)
    indx = torch.empty((n, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((n, k), dtype=torch.bfloat16, device="cuda")
    meta = moe.empty_meta(n * k, E_loc, "cuda")
    if gate:
        out = moe.forward_gate(x, dev_bf16(w_gate), w13, w2, k, params, ws, topk=(indx, vals),
                               meta=meta)
    else:
        out = moe.forward(x, dev(h["logits"]), w13, w2, k, params, ws, topk=(indx, vals),
                          meta=meta)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    ind = indx.cpu().numpy()
    if not gate:
        ref_i, ref_v = oracle.route(h["logits"], k, case.gating)
        np.testing.assert_array_equal(ind, ref_i)
        assert np.abs(host_bits(vals).astype(np.int32) - ref_v.astype(np.int32)).max() <= 1
    ref_m = oracle.metadata(ind, host_bits(vals), E, expert_map=m, n_local=E_loc)
    kept = int(ref_m["offs"][-1])
    for key in ("col_sum", "offs", "row_sorted"):
        np.testing.assert_array_equal(meta[key].cpu().numpy(), ref_m[key], err_msg=key)
    np.testing.assert_array_equal(meta["col_sorted"].cpu().numpy()[:kept], ref_m["col_sorted"])
    np.testing.assert_array_equal(host_bits(meta["gate_scal"])[:kept], ref_m["gate_scal"])
    ref = oracle.ffn(h["x"], ind, host_bits(vals), h["w13"][inv], h["w2"][inv], expert_map=m,
                     n_experts=E, act=case.act, layout=case.layout)
    got = host_bits(out)
    none_local = (m[ind] < 0).all(axis=1)
    assert not got[none_local].any(), "tokens without a local slot must give zero rows"
    if (~none_local).any():
        assert_layer_close(got[~none_local], ref[~none_local], case.name)
    return ref_m, none_local


@pytest.mark.parametrize("n,E,k,ranks,r", [
    (3, 32, 4, 4, 1),       # one-CTA decode kernel, fused gather (n*k <= 2 E_loc)
    (64, 32, 4, 2, 0),      # cooperative kernel, decode tiling
    (4096, 32, 4, 4, 3),    # cooperative kernel over all SMs, 256-row token tiles
])
def test_gptoss_shaped_rank(n, E, k, ranks, r):
    case = I.LayerCase(f"ep_n{n}", n=n, H=256, E=E, k=k, I=128, act="swiglu_oai",
                       layout="interleaved", w_std=0.05, seed=n)
    m, inv = _rank_map(E, ranks, r)
    ref_m, none_local = _run(case, m, inv)
    assert ref_m["offs"][-1] > 0 and (ref_m["row_sorted"] == -1).any()


def test_rank_on_the_tokens_on_m_kernel():
    """The same contract through the tokens-on-M grouped GEMM (X_sorted from
    the routing kernel's row copy, which skips dropped slots)."""
    case = I.LayerCase("ep_tiled", n=700, H=256, E=16, k=4, I=128, act="swiglu_oai",
                       layout="interleaved", w_std=0.05, seed=17)
    m, inv = _rank_map(16, 2, 1, permute=True)
    _run(case, m, inv, ffn_kernel="tiled")


def test_top1_rank_through_the_combine():
    """k = 1 with a map: the w2 epilogue cannot write the output directly (a
    token on another rank needs a zero row), so the combine runs."""
    case = I.LayerCase("ep_top1", n=1000, H=128, E=8, k=1, I=256, gating="softmax_all",
                       act="swiglu", layout="packed", w_std=0.05, seed=7)
    m, inv = _rank_map(8, 2, 1, permute=True)
    _, none_local = _run(case, m, inv)
    assert none_local.any() and (~none_local).any()


def test_router_matmul_rank():
    case = I.LayerCase("ep_gate", n=300, H=256, E=16, k=2, I=128, act="swiglu",
                       layout="interleaved", w_std=0.05, seed=11)
    m, inv = _rank_map(16, 4, 2, permute=True)
    _run(case, m, inv, gate=True)


def test_no_local_expert_gives_zeros():
    case = I.LayerCase("ep_none", n=50, H=128, E=8, k=2, I=128, act="swiglu_oai",
                       layout="interleaved", w_std=0.05, seed=3)
    m = np.full(8, -1, dtype=np.int32)
    inv = np.array([0])
    ref_m, none_local = _run(case, m, inv)
    assert ref_m["offs"][-1] == 0 and none_local.all()


def test_ranks_add_up_to_the_full_layer():
    """Two ranks' outputs (bf16) add up to the single-GPU layer output within
    the layer tolerance: expert parallelism splits the same sum."""
    case = I.LayerCase("ep_sum", n=200, H=256, E=8, k=2, I=128, act="swiglu_oai",
                       layout="interleaved", w_std=0.05, seed=5)
    h = I.layer_inputs(case)
    x, logits = dev_bf16(h["x"]), dev(h["logits"])
    full = moe.forward(x, logits, dev_bf16(h["w13"]), dev_bf16(h["w2"]), case.k,
                       moe.make_params(case.gating, case.act, case.layout),
                       moe.workspace(case.n, case.E, case.k, case.H, case.I))
    total = torch.zeros((case.n, case.H), dtype=torch.float32, device="cuda")
    for r in range(2):
        m, inv = _rank_map(8, 2, r)
        emap = dev(m)
        params = moe.make_params(case.gating, case.act, case.layout, expert_map=emap,
                                 n_local_experts=inv.size)
        part = moe.forward(x, logits, dev_bf16(h["w13"][inv]), dev_bf16(h["w2"][inv]), case.k,
                           params, moe.workspace(case.n, case.E, case.k, case.H, case.I))
        total += part.float()
    torch.cuda.synchronize()
    assert_layer_close(host_bits(total.to(torch.bfloat16)), host_bits(full), "sum of ranks")


@pytest.mark.parametrize("n", [3, 600])  # the one-CTA decode kernel, the cooperative one
def test_map_entries_outside_the_local_range_flag_invalid_arg(n):
    """An entry outside [-1, n_local) counts as -1 (its slots are dropped) and
    records MOE_ERR_INVALID_ARG in the workspace status word; the metadata
    is the oracle's with that entry set to -1."""
    case = I.LayerCase(f"ep_bad_n{n}", n=n, H=128, E=8, k=2, I=128, act="swiglu",
                       layout="interleaved", w_std=0.05, seed=n)
    h = I.layer_inputs(case)
    m, inv = _rank_map(8, 2, 0)              # experts 0..3 local
    ref_i, ref_v = oracle.route(h["logits"], case.k)
    bad_e = int(ref_i[0, 0])                 # an expert that receives a slot
    m_bad = m.copy()
    m_bad[bad_e] = inv.size                  # one past the local range
    m_ref = m.copy()
    m_ref[bad_e] = -1
    emap = dev(m_bad)
    params = moe.make_params(case.gating, case.act, case.layout, expert_map=emap,
                             n_local_experts=inv.size)
    ws = moe.workspace(n, case.E, case.k, case.H, case.I)
    indx = torch.empty((n, case.k), dtype=torch.int32, device="cuda")
    vals = torch.empty((n, case.k), dtype=torch.bfloat16, device="cuda")
    meta = moe.empty_meta(n * case.k, inv.size, "cuda")
    moe.forward(dev_bf16(h["x"]), dev(h["logits"]), dev_bf16(h["w13"][inv]),
                dev_bf16(h["w2"][inv]), case.k, params, ws, topk=(indx, vals), meta=meta)
    assert moe.read_status(ws, reset=True) == 1  # MOE_ERR_INVALID_ARG
    ref_m = oracle.metadata(indx.cpu().numpy(), host_bits(vals), case.E, expert_map=m_ref,
                            n_local=inv.size)
    for key in ("col_sum", "offs", "row_sorted"):
        np.testing.assert_array_equal(meta[key].cpu().numpy(), ref_m[key], err_msg=key)
