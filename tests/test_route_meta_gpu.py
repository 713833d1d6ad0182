"""Routing and metadata on the GPU against the CPU oracle, bit for bit.

Shapes: the routing sweep n in {1, 33, 512, 4096, 16384} x (E, k) in
{(32, 4), (128, 4)} of the first report's parity test (关键源码片段,
test_routing_data_from_sparse_topk_parity), plus tie-heavy logits, both
gatings, edge values of E and k, multi-round CTAs and degenerate routings.
Top-k indices, col_sum, offs, col_sorted, row_sorted and gate_scal must
match exactly; gate weights (fp32 softmax on the GPU, float64 in the oracle,
both rounded to bf16) may differ by one bf16 ulp on rare rounding ties."""
import numpy as np
import pytest
import torch

import mixture_experts_routing_warp_gb300 as moe
import oracle
import moe_inputs as I

from helpers import dev, host_bits

pytestmark = pytest.mark.gpu


def _gpu_route(logits, k, gating="softmax_topk"):
    indx, vals = moe.route(dev(logits), k, gating)
    return indx, vals


def _check_vals(got_bits, ref_bits):
    d = np.abs(got_bits.astype(np.int32) - ref_bits.astype(np.int32))
    assert d.max(initial=0) <= 1, d.max()
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= 1e-3, frac


def _check_meta(indx, vals, E):
    n, k = indx.shape
    ws = moe.workspace(max(n, 1), E, k, 64, 64)
    m = moe.build_metadata(indx, vals, E, ws)
    torch.cuda.synchronize()
    assert moe.read_status(ws) == 0
    ref = oracle.metadata(indx.cpu().numpy(), host_bits(vals), E)
    for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
        np.testing.assert_array_equal(m[key].cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(host_bits(m["gate_scal"]), ref["gate_scal"])
    return m


@pytest.mark.parametrize("n", I.ROUTE_SWEEP_N)
@pytest.mark.parametrize("E,k", I.ROUTE_SWEEP_EK)
@pytest.mark.parametrize("tie_heavy", [False, True])
def test_routing_sweep_bit_exact(n, E, k, tie_heavy):
    logits = I.route_logits(n, E, seed=0, tie_heavy=tie_heavy)
    ref_i, ref_v = oracle.route(logits, k)
    indx, vals = _gpu_route(logits, k)
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
    _check_vals(host_bits(vals), ref_v)
    _check_meta(indx, vals, E)


@pytest.mark.parametrize("E,k", [(1, 1), (2, 2), (7, 3), (33, 8), (64, 1), (256, 8), (256, 1),
                                 (100, 5)])
@pytest.mark.parametrize("gating", ["softmax_topk", "softmax_all"])
def test_routing_shapes_and_gatings(E, k, gating):
    n = 777
    for logits in (I.route_logits(n, E, seed=3), I.small_int_logits(n, E, seed=3, levels=2)):
        ref_i, ref_v = oracle.route(logits, k, gating)
        indx, vals = _gpu_route(logits, k, gating)
        np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
        _check_vals(host_bits(vals), ref_v)
        _check_meta(indx, vals, E)


def test_signed_zero_ties_and_negative_logits():
    logits = np.array([[-0.0, 0.0, -1.0, -1.0], [0.0, -0.0, -3.0, -0.5],
                       [-5.0, -5.0, -5.0, -5.0]], dtype=np.float32)
    indx, _ = _gpu_route(logits, 3)
    ref_i, _ = oracle.route(logits, 3)
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)


def test_many_rounds_per_cta():
    """2e5 tokens x top-8: more slots than one round per CTA can hold."""
    n, E, k = 200_000, 64, 8
    logits = I.route_logits(n, E, seed=11)
    indx, vals = _gpu_route(logits, k)
    ref_i, _ = oracle.route(logits, k)
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
    _check_meta(indx, vals, E)


@pytest.mark.parametrize("pattern", ["one_expert", "last_expert", "round_robin", "random"])
def test_metadata_degenerate_routings(pattern):
    n, E, k = 5000, 16, 4
    rng = np.random.default_rng(5)
    if pattern == "one_expert":
        # not a valid top-k (repeats) but a valid histogram input: all slots to expert 0
        ind = np.zeros((n, k), np.int32)
    elif pattern == "last_expert":
        ind = np.full((n, k), E - 1, np.int32)
    elif pattern == "round_robin":
        ind = (np.arange(n * k, dtype=np.int32) % E).reshape(n, k)
    else:
        ind = rng.integers(0, E, size=(n, k)).astype(np.int32)
    vals = I.f32_to_bf16_bits(rng.random((n, k), dtype=np.float32))
    indx = dev(ind)
    v = torch.from_numpy(vals.view(np.int16)).view(torch.bfloat16).cuda()
    _check_meta(indx, v, E)


def test_empty_input_is_a_noop():
    logits = torch.empty((0, 32), dtype=torch.float32, device="cuda")
    indx, vals = moe.route(logits, 4)
    assert indx.shape == (0, 4)
    ws = moe.workspace(1, 32, 4, 64, 64)
    m = moe.build_metadata(indx, vals, 32, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(m["col_sum"].cpu().numpy(), np.zeros(32))
    np.testing.assert_array_equal(m["offs"].cpu().numpy(), np.zeros(33))
    assert moe.read_status(ws) == 0


def test_run_to_run_bit_identical():
    logits = I.route_logits(16384, 128, seed=1, tie_heavy=True)
    a = _gpu_route(logits, 4)
    ws = moe.workspace(16384, 128, 4, 64, 64)
    ma = {k: v.clone() for k, v in moe.build_metadata(*a, 128, ws).items()}
    for _ in range(3):
        b = _gpu_route(logits, 4)
        mb = moe.build_metadata(*b, 128, ws)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int16),
                                                       b[1].view(torch.int16))
        for key in ma:
            assert torch.equal(ma[key].view(torch.int16) if ma[key].dtype == torch.bfloat16
                               else ma[key],
                               mb[key].view(torch.int16) if mb[key].dtype == torch.bfloat16
                               else mb[key]), key


@pytest.mark.parametrize("n,E,k", [(16384, 128, 4), (4096, 32, 4), (33, 8, 2), (1, 4, 1),
                                   (777, 100, 5), (5000, 7, 3), (3000, 256, 8),
                                   (600_000, 16, 4),
                                   # decode sizes (n*k <= 32): the one-CTA kernel
                                   (1, 32, 4), (8, 32, 4), (2, 256, 8), (4, 128, 8),
                                   (32, 16, 1), (5, 7, 3), (3, 100, 5), (16, 64, 2)])
@pytest.mark.parametrize("gating", ["softmax_topk", "softmax_all"])
def test_route_metadata_equals_route_then_build(n, E, k, gating):
    """The fused call (one CTA for decode sizes, one cooperative kernel when
    each SM's slots fit in shared memory, else two kernels) gives the
    two-call result bit for bit."""
    logits = dev(I.route_logits(n, E, seed=n % 97, tie_heavy=True))
    i1, v1 = moe.route(logits, k, gating)
    ws1 = moe.workspace(n, E, k, 64, 64)
    m1 = moe.build_metadata(i1, v1, E, ws1)
    i2, v2, m2 = moe.route_metadata(logits, k, gating=gating)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2)
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    for key in m1:
        a, b = m1[key], m2[key]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), key
    if n <= 20000:
        ref_i, ref_v = oracle.route(logits.cpu().numpy(), k, gating)
        np.testing.assert_array_equal(i2.cpu().numpy(), ref_i)
        ref_m = oracle.metadata(ref_i, host_bits(v2), E)
        for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
            np.testing.assert_array_equal(m2[key].cpu().numpy(), ref_m[key], err_msg=key)


@pytest.mark.parametrize("E,k", [(128, 4), (32, 4), (6, 2)])
def test_logits_base_only_4_byte_aligned(E, k):
    """The API asks only 4-byte alignment of logits: a base offset by one
    float must route exactly like an aligned copy (scalar-load path)."""
    n = 1000
    host = I.route_logits(n, E, seed=9)
    flat = torch.empty(n * E + 1, dtype=torch.float32, device="cuda")
    shifted = flat[1:].view(n, E)
    shifted.copy_(torch.from_numpy(host))
    assert shifted.data_ptr() % 16 != 0
    i1, v1 = moe.route(shifted, k)
    i2, v2 = moe.route(dev(host), k)
    i3, v3, _ = moe.route_metadata(shifted, k)
    torch.cuda.synchronize()
    assert torch.equal(i1, i2) and torch.equal(i1, i3)
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    ref_i, _ = oracle.route(host, k)
    np.testing.assert_array_equal(i1.cpu().numpy(), ref_i)


def _near_tie_logits(n, E, k, seed):
    """N(0,1) logits where, per token, an unselected expert (or one of the
    selected) is moved to within 1..300 ulps of the k-th largest value, above
    or below it, or onto it exactly: the selection then hinges on the low bits
    of the fp32 values, below the resolution of the kernels' 32-bit
    selection keys (which then fall back to exact 64-bit keys)."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((n, E)).astype(np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")
    bits = logits.view(np.uint32)
    for t in range(n):
        kth = order[t, k - 1]
        other = order[t, rng.integers(k, E)] if rng.random() < 0.7 else order[t, rng.integers(0, k)]
        if other == kth:
            continue
        step = int(rng.integers(-300, 301))
        v = np.int64(bits[t, kth])
        # move by `step` ulps in magnitude, staying on the same side of zero
        bits[t, other] = np.uint32(max(1, min(0x7F7FFFFF, (v & 0x7FFFFFFF) + step)) | (v & 0x80000000))
    return logits


@pytest.mark.parametrize("E,k", [(32, 4), (128, 4), (16, 2), (256, 4), (6, 3)])
def test_near_ties_below_the_selection_key_resolution(E, k):
    """Bit-exact top-k (ties to the lower id) when candidates differ only in
    the lowest mantissa bits, through the route kernel and the fused route +
    metadata kernel."""
    n = 4096
    logits = _near_tie_logits(n, E, k, seed=E * 10 + k)
    ref_i, ref_v = oracle.route(logits, k)
    indx, vals = _gpu_route(logits, k)
    np.testing.assert_array_equal(indx.cpu().numpy(), ref_i)
    _check_vals(host_bits(vals), ref_v)
    i2, v2, m2 = moe.route_metadata(dev(logits), k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(i2.cpu().numpy(), ref_i)
    _check_vals(host_bits(v2), ref_v)
    ref_m = oracle.metadata(ref_i, host_bits(v2), E)
    for key in ("col_sum", "offs", "col_sorted", "row_sorted"):
        np.testing.assert_array_equal(m2[key].cpu().numpy(), ref_m[key], err_msg=key)
