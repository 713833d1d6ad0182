"""Pins for the oracle's per-expert FFN and gate-weighted combine.

* the w13 / w2 contractions against numpy float64 matmul (a transposed
  operand or a wrong index fails);
* activations at hand-worked points, through selector weights that route
  chosen x entries to gate / up (a swapped gate and up fails);
* the w13 layouts as the "CuteDSL NVFP4 MoE adds SwiGLU-OAI and ReLU2"
  report defines them (关键源码片段: interleaved gate = w13[:, 0::2],
  up = w13[:, 1::2]; packed halves [gate; up]);
* SwiGLU-OAI with alpha=1, beta=0, no clamp equals SwiGLU bit for bit;
  SwiGLU with a clamp limit ("SILU + clamp", 实现拆解 and 关键源码片段: SiLU
  forwards only the limit) equals SwiGLU-OAI with alpha=1, beta=0 and that
  limit, and clamps at hand-worked points;
* the non-gated ReLU2 ("RELU2_NO_MUL", 实现拆解) at hand-worked points
  through one-row selectors, and as a dense E = 1 layer against numpy;
* the combine equals the masked per-expert index_add_ loop of the MiniMind
  issue (Summary) and the sorted dispatch ("It is removable in plain
  PyTorch") bit for bit;
* the router weight multiplies the expert output (exact power-of-two check).
"""
import math

import numpy as np
import pytest

import oracle
import moe_inputs as I

ONE = 0x3F80  # bf16 1.0


def _b(v):
    return I.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def test_contractions_against_numpy_float64():
    rng = np.random.default_rng(0)
    H, Idim = 96, 40
    x = _b(rng.standard_normal(H))
    w13 = _b(rng.standard_normal((2 * Idim, H)) * 0.1)
    w2 = _b(rng.standard_normal((H, Idim)) * 0.1)
    for act in ("swiglu", "swiglu_oai"):
        a, h, y = oracle.expert_row(x, w13, w2, act=act)
        a_ref = oracle.bf16_to_f64(w13) @ oracle.bf16_to_f64(x)
        scale = np.abs(oracle.bf16_to_f64(w13)) @ np.abs(oracle.bf16_to_f64(x))
        assert np.all(np.abs(a - a_ref) <= 1e-13 * scale + 1e-300)
        y_ref = oracle.bf16_to_f64(w2) @ oracle.bf16_to_f64(h)
        scale = np.abs(oracle.bf16_to_f64(w2)) @ np.abs(oracle.bf16_to_f64(h))
        assert np.all(np.abs(y - y_ref) <= 1e-13 * scale + 1e-300)


def _selector_expert(H, Idim, gate_src, up_src, layout):
    """w13 whose gate row i picks x[gate_src[i]] and up row i picks x[up_src[i]];
    w2 = identity on the first Idim outputs, so y[i] = h[i]."""
    w13 = np.zeros((2 * Idim, H), dtype=np.uint16)
    for i in range(Idim):
        g_row, u_row = (i, Idim + i) if layout == "packed" else (2 * i, 2 * i + 1)
        w13[g_row, gate_src[i]] = ONE
        w13[u_row, up_src[i]] = ONE
    w2 = np.zeros((H, Idim), dtype=np.uint16)
    for i in range(Idim):
        w2[i, i] = ONE
    return w13, w2


def _silu(g):
    return g / (1.0 + math.exp(-g))


@pytest.mark.parametrize("layout", ["packed", "interleaved"])
def test_swiglu_at_worked_points(layout):
    xs = [2.0, 3.0, 0.0, -1.5, 5.0, 1.0, -4.0, 0.5]
    x = _b(xs)
    pairs = [(0, 1), (1, 0), (2, 4), (4, 2), (3, 5), (6, 7)]  # (gate entry, up entry)
    w13, w2 = _selector_expert(8, len(pairs), [p[0] for p in pairs], [p[1] for p in pairs],
                               layout)
    _, h, y = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout)
    expected = [_silu(xs[g]) * xs[u] for g, u in pairs]
    np.testing.assert_array_equal(h, oracle.f64_to_bf16(np.array(expected)))
    # hand-worked: silu(2)*3 = 5.2848 and silu(3)*2 = 5.7154 round to different bf16
    assert oracle.bf16_to_f64(h[:2]).tolist() == [5.28125, 5.71875]
    assert h[2] == 0 and h[3] == 0  # silu(0) = 0, and up = 0
    np.testing.assert_array_equal(oracle.f64_to_bf16(y[:len(pairs)]), h)


@pytest.mark.parametrize("layout", ["packed", "interleaved"])
def test_swiglu_oai_clamps_at_worked_points(layout):
    xs = [10.0, -9.0, 9.0, 7.0, -7.0, 0.5, -3.0, 2.0]
    x = _b(xs)
    pairs = [(0, 1), (0, 2), (3, 4), (5, 6), (6, 7), (1, 5)]
    w13, w2 = _selector_expert(8, len(pairs), [p[0] for p in pairs], [p[1] for p in pairs],
                               layout)
    _, h, _ = oracle.expert_row(x, w13, w2, act="swiglu_oai", layout=layout)

    def oai(g, u, alpha=1.702, beta=1.0, limit=7.0):
        g = min(g, limit)
        u = max(-limit, min(u, limit))
        return (u + beta) * g / (1.0 + math.exp(-alpha * g))

    expected = [oai(xs[g], xs[u]) for g, u in pairs]
    np.testing.assert_array_equal(h, oracle.f64_to_bf16(np.array(expected)))
    # gate 10 clamps to 7 and up -9 clamps to -7: (-7 + 1) * 7 * sigmoid(11.914) = -41.9997 -> -42
    assert oracle.bf16_to_f64(h[0]) == -42.0
    # gate clamped to 7, up 9 clamped to 7: 8 * 7 * sigmoid(11.914) -> 56
    assert oracle.bf16_to_f64(h[1]) == 56.0
    # gate -9 is not clamped from below: (0.5 + 1) * -9 * sigmoid(-15.3) ~ -3e-6
    assert -1e-5 < oracle.bf16_to_f64(h[5]) < 0


def test_parameters_override_defaults():
    rng = np.random.default_rng(1)
    H, Idim = 32, 16
    x = _b(rng.standard_normal(H) * 4)
    w13 = _b(rng.standard_normal((2 * Idim, H)))
    w2 = _b(rng.standard_normal((H, Idim)) * 0.1)
    base = oracle.expert_row(x, w13, w2, act="swiglu_oai")[1]
    same = oracle.expert_row(x, w13, w2, act="swiglu_oai", alpha=1.702, beta=1.0, limit=7.0)[1]
    np.testing.assert_array_equal(base, same)
    for kw in ({"alpha": 1.0}, {"beta": 0.0}, {"limit": 3.0}):
        assert not np.array_equal(base, oracle.expert_row(x, w13, w2, act="swiglu_oai", **kw)[1])


def test_oai_reduces_to_swiglu():
    rng = np.random.default_rng(2)
    H, Idim = 64, 48
    x = _b(rng.standard_normal(H) * 3)
    w13 = _b(rng.standard_normal((2 * Idim, H)) * 0.3)
    w2 = _b(rng.standard_normal((H, Idim)) * 0.1)
    for layout in ("packed", "interleaved"):
        s = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout)
        o = oracle.expert_row(x, w13, w2, act="swiglu_oai", layout=layout, alpha=1.0,
                              beta=0.0, limit=math.inf)
        np.testing.assert_array_equal(s[1], o[1])
        np.testing.assert_array_equal(s[2], o[2])


def _interleave(w13_packed):
    E, I2, H = w13_packed.shape
    Idim = I2 // 2
    out = np.empty_like(w13_packed)
    out[:, 0::2] = w13_packed[:, :Idim]
    out[:, 1::2] = w13_packed[:, Idim:]
    return out


@pytest.mark.parametrize("act", ["swiglu", "swiglu_oai"])
def test_layout_invariance(act):
    case = I.TINY
    d = I.layer_inputs(case)
    indx, vals = oracle.route(d["logits"], case.k)
    a = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], act=act, layout="packed")
    b = oracle.ffn(d["x"], indx, vals, _interleave(d["w13"]), d["w2"], act=act,
                   layout="interleaved")
    np.testing.assert_array_equal(a, b)


def _tiny(act="swiglu", gating="softmax_topk", n=33, E=8, k=2):
    case = I.LayerCase("t", n=n, H=64, E=E, k=k, I=128, gating=gating, act=act)
    d = I.layer_inputs(case)
    indx, vals = oracle.route(d["logits"], k, gating)
    return case, d, indx, vals


@pytest.mark.parametrize("act", ["swiglu", "swiglu_oai"])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_combine_equals_masked_per_expert_loop(act, k):
    case, d, indx, vals = _tiny(act=act, k=k)
    out, y_slot, _ = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], act=act,
                                want_slots=True)
    # masked loop: for each expert in turn, every token that picked it,
    # y[t] += expert(x[t]) * weight   (accumulated in float64)
    acc = np.zeros((case.n, case.H))
    for e in range(case.E):
        tok, slot = np.nonzero(indx == e)
        for t, j in zip(tok, slot):
            _, _, y = oracle.expert_row(d["x"][t], d["w13"][e], d["w2"][e], act=act)
            acc[t] += y * oracle.bf16_to_f64(vals[t, j])
    np.testing.assert_array_equal(out, oracle.f64_to_bf16(acc))


@pytest.mark.parametrize("k", [1, 3])
def test_combine_equals_sorted_dispatch(k):
    case, d, indx, vals = _tiny(k=k, E=6)
    m = oracle.metadata(indx, vals, case.E)
    out = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"])
    # sorted dispatch: row p is token col_sorted[p] // k for expert of segment p
    y_flat = np.zeros((case.n * k, case.H))
    for e in range(case.E):
        for p in range(m["offs"][e], m["offs"][e + 1]):
            f = m["col_sorted"][p]
            _, _, y = oracle.expert_row(d["x"][f // k], d["w13"][e], d["w2"][e])
            y_flat[f] = y * oracle.bf16_to_f64(m["gate_scal"][p])     # scatter
    acc = np.zeros((case.n, case.H))
    for t in range(case.n):
        for j in np.argsort(indx[t]):   # ascending expert id
            acc[t] += y_flat[t * k + j]
    np.testing.assert_array_equal(out, oracle.f64_to_bf16(acc))


def test_weight_multiplies_the_expert_output():
    case, d, indx, vals = _tiny(k=1)
    half = np.full_like(vals, 0x3F00)   # 0.5
    one = np.full_like(vals, ONE)
    o1 = oracle.bf16_to_f64(oracle.ffn(d["x"], indx, one, d["w13"], d["w2"]))
    oh = oracle.bf16_to_f64(oracle.ffn(d["x"], indx, half, d["w13"], d["w2"]))
    np.testing.assert_array_equal(oh, o1 * 0.5)  # exact: scaling after the nonlinearity
    zero = np.zeros_like(vals)
    assert not oracle.ffn(d["x"], indx, zero, d["w13"], d["w2"]).any()


def test_single_expert_layer_against_numpy():
    """E = 1, k = 1: every token goes to the one expert with gate weight 1,
    so the layer is a dense SwiGLU MLP: bf16(W2 . bf16(silu(W1 x) * (W3 x)))."""
    case = I.LayerCase("dense", n=40, H=64, E=1, k=1, I=96)
    d = I.layer_inputs(case)
    indx, vals = oracle.route(d["logits"], 1)
    assert (vals == ONE).all() and (indx == 0).all()
    out = oracle.bf16_to_f64(oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"]))
    x = oracle.bf16_to_f64(d["x"])
    w13 = oracle.bf16_to_f64(d["w13"][0])
    w2 = oracle.bf16_to_f64(d["w2"][0])
    a = x @ w13.T
    g, u = a[:, :case.I], a[:, case.I:]
    h = oracle.bf16_to_f64(oracle.f64_to_bf16(g / (1 + np.exp(-g)) * u))
    ref = h @ w2.T
    err = np.abs(out - ref)
    # out is ref rounded once to bf16 (h may flip one bf16 ulp where numpy's
    # summation order lands on the other side of a rounding boundary)
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9)
    assert np.all(err <= 3 * half_ulp), (err / half_ulp).max()
    assert (err <= half_ulp * (1 + 1e-9)).mean() > 0.99


def test_token_subset_matches_full_run():
    case, d, indx, vals = _tiny(act="swiglu_oai", k=2)
    full = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], act="swiglu_oai")
    toks = np.array([32, 0, 7, 7, 19])
    sub = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], tokens=toks, act="swiglu_oai")
    np.testing.assert_array_equal(sub, full[toks])


def test_thread_count_does_not_change_bits(monkeypatch):
    import subprocess, sys, os
    code = ("import sys; sys.path.insert(0, '.'); import oracle, numpy as np;"
            "import moe_inputs as I;"
            "c = I.TINY; d = I.layer_inputs(c); i, v = oracle.route(d['logits'], c.k);"
            "print(oracle.ffn(d['x'], i, v, d['w13'], d['w2']).tobytes().hex())")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for threads in ("1", "3"):
        env = dict(os.environ, OMP_NUM_THREADS=threads)
        outs.append(subprocess.run([sys.executable, "-c", code], cwd=root, env=env,
                                   capture_output=True, text=True, check=True).stdout)
    assert outs[0] == outs[1]


@pytest.mark.parametrize("layout", ["packed", "interleaved"])
def test_swiglu_clamp_at_worked_points(layout):
    xs = [10.0, -9.0, 9.0, 2.0, -3.0, 0.5, 1.0, -1.0]
    x = _b(xs)
    pairs = [(0, 1), (0, 2), (3, 2), (4, 5), (1, 6), (6, 7)]
    w13, w2 = _selector_expert(8, len(pairs), [p[0] for p in pairs], [p[1] for p in pairs],
                               layout)
    _, h, _ = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout, limit=3.0)

    def silu_clamp(g, u, limit=3.0):
        g = min(g, limit)
        u = max(-limit, min(u, limit))
        return _silu(g) * u

    expected = [silu_clamp(xs[g], xs[u]) for g, u in pairs]
    np.testing.assert_array_equal(h, oracle.f64_to_bf16(np.array(expected)))
    # gate 10 -> 3 and up -9 -> -3: silu(3) * -3 = -8.5732 -> bf16 -8.5625
    assert oracle.bf16_to_f64(h[0]) == -8.5625
    # gate 10 -> 3 and up 9 -> 3: +8.5625; gate 2 stays, up 9 -> 3: silu(2)*3 = 5.2848 -> 5.28125
    assert oracle.bf16_to_f64(h[1]) == 8.5625 and oracle.bf16_to_f64(h[2]) == 5.28125
    # the gate is not clamped from below: silu(-9) * 1 ~ -1.1e-3
    assert -2e-3 < oracle.bf16_to_f64(h[4]) < -1e-3
    # without the limit the same inputs differ (the clamp acts)
    _, h_free, _ = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout)
    assert not np.array_equal(h, h_free)


def test_swiglu_clamp_equals_oai_with_unit_alpha_zero_beta():
    rng = np.random.default_rng(5)
    H, Idim = 64, 48
    x = _b(rng.standard_normal(H) * 3)
    w13 = _b(rng.standard_normal((2 * Idim, H)) * 0.5)
    w2 = _b(rng.standard_normal((H, Idim)) * 0.1)
    for layout in ("packed", "interleaved"):
        for limit in (0.5, 2.0, 7.0):
            s = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout, limit=limit)
            o = oracle.expert_row(x, w13, w2, act="swiglu_oai", layout=layout, alpha=1.0,
                                  beta=0.0, limit=limit)
            np.testing.assert_array_equal(s[1], o[1])
            np.testing.assert_array_equal(s[2], o[2])


def test_relu2_at_worked_points():
    xs = [3.0, -2.0, 0.5, 0.0, -0.25, 1.5, 4.0, -8.0]
    x = _b(xs)
    H, Idim = 8, 8
    w1 = np.zeros((Idim, H), dtype=np.uint16)   # non-gated: I rows, row i picks x[src[i]]
    src = [0, 1, 2, 3, 4, 5, 6, 7]
    for i, j in enumerate(src):
        w1[i, j] = ONE
    w2 = np.zeros((H, Idim), dtype=np.uint16)
    for i in range(Idim):
        w2[i, i] = ONE
    a, h, y = oracle.expert_row(x, w1, w2, act="relu2")
    assert a.shape == (Idim,)
    # max(v, 0)^2, all exact in bf16: 9, 0, 0.25, 0, 0, 2.25, 16, 0
    assert oracle.bf16_to_f64(h).tolist() == [9.0, 0.0, 0.25, 0.0, 0.0, 2.25, 16.0, 0.0]
    np.testing.assert_array_equal(oracle.f64_to_bf16(y), h)
    # two picks summed before the activation: (3 + -2)^2 = 1, (-2 + 0.5) -> 0
    w1b = np.zeros((2, H), dtype=np.uint16)
    w1b[0, 0] = w1b[0, 1] = ONE
    w1b[1, 1] = w1b[1, 2] = ONE
    _, hb, _ = oracle.expert_row(x, w1b, np.zeros((H, 2), dtype=np.uint16), act="relu2")
    assert oracle.bf16_to_f64(hb).tolist() == [1.0, 0.0]


def test_relu2_rejects_a_clamp_limit():
    with pytest.raises(ValueError):
        oracle.act_params(act="relu2", limit=3.0)


def test_single_expert_relu2_layer_against_numpy():
    """E = 1, k = 1, ReLU2: a dense non-gated MLP, bf16(W2 . bf16(max(W1 x, 0)^2))."""
    case = I.LayerCase("dense_relu2", n=40, H=64, E=1, k=1, I=96, act="relu2")
    d = I.layer_inputs(case)
    assert d["w13"].shape == (1, case.I, case.H)
    indx, vals = oracle.route(d["logits"], 1)
    out = oracle.bf16_to_f64(oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], act="relu2"))
    x = oracle.bf16_to_f64(d["x"])
    a = x @ oracle.bf16_to_f64(d["w13"][0]).T
    h = oracle.bf16_to_f64(oracle.f64_to_bf16(np.maximum(a, 0.0) ** 2))
    ref = h @ oracle.bf16_to_f64(d["w2"][0]).T
    err = np.abs(out - ref)
    half_ulp = np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9)
    assert np.all(err <= 3 * half_ulp), (err / half_ulp).max()
    assert (err <= half_ulp * (1 + 1e-9)).mean() > 0.99


@pytest.mark.parametrize("k", [1, 2])
def test_relu2_combine_equals_masked_per_expert_loop(k):
    case = I.LayerCase("t_relu2", n=33, H=64, E=8, k=k, I=128, act="relu2")
    d = I.layer_inputs(case)
    indx, vals = oracle.route(d["logits"], k)
    out = oracle.ffn(d["x"], indx, vals, d["w13"], d["w2"], act="relu2")
    acc = np.zeros((case.n, case.H))
    for e in range(case.E):
        tok, slot = np.nonzero(indx == e)
        for t, j in zip(tok, slot):
            _, _, y = oracle.expert_row(d["x"][t], d["w13"][e], d["w2"][e], act="relu2")
            acc[t] += y * oracle.bf16_to_f64(vals[t, j])
    np.testing.assert_array_equal(out, oracle.f64_to_bf16(acc))
