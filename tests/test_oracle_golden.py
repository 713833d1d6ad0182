"""Oracle against the stored fixtures in tests/golden/.

* swiglu_oai_defaults.txt and w13_layouts.txt hold facts printed on the
  pages (cited in each file);
* tiny_layer_oracle.txt holds the oracle's own outputs for the tiny layer,
  written by tests/golden/make_golden.py: a regression anchor, not an
  independent pin."""
import math
import os

import numpy as np

import oracle
import moe_inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _kv(name):
    out = {}
    for ln in open(os.path.join(GOLDEN, name)):
        if ln.strip() and not ln.startswith("#"):
            key, *rest = ln.split()
            out[key] = rest
    return out


def test_swiglu_oai_defaults_from_the_page():
    kv = _kv("swiglu_oai_defaults.txt")
    assert (oracle.OAI_ALPHA, oracle.OAI_BETA, oracle.OAI_LIMIT) == (
        float(kv["alpha"][0]), float(kv["beta"][0]), float(kv["limit"][0]))
    p = oracle.act_params("swiglu_oai")
    assert (p.alpha, p.beta, p.limit) == (1.702, 1.0, 7.0)
    s = oracle.act_params("swiglu")       # plain SwiGLU gets no clamp
    assert math.isinf(s.limit)


def test_w13_layouts_from_the_page():
    kv = _kv("w13_layouts.txt")
    Idim, H = 3, 8
    for layout in ("interleaved", "packed"):
        roles = kv[layout]
        # row r of w13 picks x[r]; x[r] = r + 1, so a[r] = r + 1
        w13 = np.zeros((2 * Idim, H), dtype=np.uint16)
        for r in range(2 * Idim):
            w13[r, r] = 0x3F80
        w2 = np.zeros((H, Idim), dtype=np.uint16)
        x = I.f32_to_bf16_bits(np.arange(1, H + 1, dtype=np.float32))
        _, h, _ = oracle.expert_row(x, w13, w2, act="swiglu", layout=layout)
        for i in range(Idim):
            g = float(roles.index(f"gate{i}") + 1)
            u = float(roles.index(f"up{i}") + 1)
            want = oracle.f64_to_bf16(np.array([g / (1 + math.exp(-g)) * u]))[0]
            assert h[i] == want, (layout, i)


def test_tiny_layer_regression():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(GOLDEN, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    stored = mg.load()
    now = mg.compute()
    assert stored.keys() == now.keys()
    for key in stored:
        np.testing.assert_array_equal(stored[key], now[key], err_msg=key)
