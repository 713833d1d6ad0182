"""The router matmul fused with the top-k (moe_route_gemm, moe_forward_gate)
against the oracle, on the GPU through the C ABI.

The "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward" report
(功能与动机) names the fusion of the router with expert selection (issue
#28986) as the next step after its own change. The kernel's fp32 logits
must match the oracle's float64 router matmul within fp32 accumulation
error; its top-k must equal, bit for bit, the oracle's routing of those same
logits (the same tie rule), with gate weights within one bf16 ulp; and the
whole layer from x and the gate weights must match the oracle's layer on
that routing."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import oracle
import moe_inputs as I

from helpers import assert_layer_close, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

CASES = [
    # n, E, H, k, gating
    (33, 8, 64, 2, "softmax_topk"),
    (1, 32, 2880, 4, "softmax_topk"),       # GPT-OSS router, decode
    (300, 32, 2880, 4, "softmax_topk"),     # GPT-OSS router, ragged 128-row tail
    (4096, 4, 512, 1, "softmax_all"),       # MiniMind router
    (1000, 16, 512, 1, "softmax_all"),
    (257, 128, 1024, 4, "softmax_topk"),
    (130, 256, 256, 8, "softmax_topk"),     # E = 256, k = 8
    (64, 40, 128, 3, "softmax_all"),        # E not a multiple of 32
]


@pytest.mark.parametrize("n,E,H,k,gating", CASES)
def test_route_gemm_matches_oracle(n, E, H, k, gating):
    case = I.LayerCase(f"router_n{n}_e{E}", n=n, H=H, E=E, k=k, I=64, gating=gating, seed=n)
    hx, hw = I.layer_x(case), I.router_weight(case)
    x, wg = dev_bf16(hx), dev_bf16(hw)
    logits = torch.empty((n, E), dtype=torch.float32, device="cuda")
    ws = moe.workspace(n, E, k, 64, 64)
    indx, vals = moe.route_gemm(x, wg, k, gating, ws=ws, logits=logits)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    got = logits.cpu().numpy()

    ref = oracle.router_logits(hx, hw, as_f32=False)
    scale = np.abs(oracle.bf16_to_f64(hx)) @ np.abs(oracle.bf16_to_f64(hw)).T
    assert np.all(np.abs(got - ref) <= 2e-4 * scale + 1e-30), np.abs(got - ref).max()

    ref_i, ref_v = oracle.route(got, k, gating)          # the same logits, the oracle's routing
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
    d = np.abs(host_bits(vals).astype(np.int32) - ref_v.astype(np.int32))
    assert d.max(initial=0) <= 1
    # the logits-input router on these logits picks the same experts
    i2, _ = moe.route(logits, k, gating)
    torch.cuda.synchronize()
    assert torch.equal(i2, indx)


def test_route_gemm_without_logits_output():
    case = I.LayerCase("router_nolog", n=200, H=512, E=64, k=4, I=64, seed=3)
    x, wg = dev_bf16(I.layer_x(case)), dev_bf16(I.router_weight(case))
    logits = torch.empty((case.n, case.E), dtype=torch.float32, device="cuda")
    a_i, a_v = moe.route_gemm(x, wg, case.k, logits=logits)
    b_i, b_v = moe.route_gemm(x, wg, case.k)
    torch.cuda.synchronize()
    assert torch.equal(a_i, b_i) and torch.equal(a_v.view(torch.int16), b_v.view(torch.int16))


@pytest.mark.parametrize("act,layout", [("swiglu_oai", "interleaved"), ("swiglu", "packed")])
def test_forward_gate_layer(act, layout):
    case = I.LayerCase("gate_layer", n=150, H=256, E=16, k=4, I=256, act=act, layout=layout,
                       w_std=0.05, seed=9)
    h = I.layer_inputs(case)
    hw = I.router_weight(case)
    x, wg = dev_bf16(h["x"]), dev_bf16(hw)
    w13, w2 = dev_bf16(h["w13"]), dev_bf16(h["w2"])
    params = moe.make_params(case.gating, act, layout)
    ws = moe.workspace(case.n, case.E, case.k, case.H, case.I)
    indx = torch.empty((case.n, case.k), dtype=torch.int32, device="cuda")
    vals = torch.empty((case.n, case.k), dtype=torch.bfloat16, device="cuda")
    meta = moe.empty_meta(case.n * case.k, case.E, "cuda")
    out = moe.forward_gate(x, wg, w13, w2, case.k, params, ws, topk=(indx, vals), meta=meta)
    r_i, r_v = moe.route_gemm(x, wg, case.k)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    assert torch.equal(indx, r_i) and torch.equal(vals.view(torch.int16), r_v.view(torch.int16))
    ind = indx.cpu().numpy()
    ref_m = oracle.metadata(ind, host_bits(vals), case.E)
    for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
        np.testing.assert_array_equal(meta[key].cpu().numpy(), ref_m[key], err_msg=key)
    ref = oracle.ffn(h["x"], ind, host_bits(vals), h["w13"], h["w2"], act=act, layout=layout)
    assert_layer_close(host_bits(out), ref, "forward_gate")
