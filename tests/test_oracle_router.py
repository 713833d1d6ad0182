"""Pins for the oracle's router matmul (logits = x . w_gate^T), the step
before routing that the "Reuse topk SparseMatrix routing metadata in GPT-OSS
MoE forward" report (功能与动机) names as the fusion issue #28986 asks for:

* brute force in pure Python on tiny inputs (the same summation order, so
  bit for bit);
* one-hot gate rows pick single entries of x exactly, and two-hot rows add
  two entries (a transposed operand or a wrong index fails);
* numpy float64 matmul within float64 rounding on a larger case;
* fp32 rounding of the float64 result is one round-to-nearest-even step.
"""
import numpy as np

import oracle
import moe_inputs as I

ONE = 0x3F80


def _b(v):
    return I.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))


def test_brute_force_tiny():
    rng = np.random.default_rng(11)
    n, E, H = 5, 4, 7
    x = _b(rng.standard_normal((n, H)))
    w = _b(rng.standard_normal((E, H)))
    got = oracle.router_logits(x, w, as_f32=False)
    xf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)
    for t in range(n):
        for e in range(E):
            s = 0.0
            for h in range(H):
                s += float(xf[t, h]) * float(wf[e, h])
            assert got[t, e] == s


def test_selector_rows():
    xs = np.array([[1.5, -2.0, 0.25, 3.0], [0.5, 4.0, -1.0, -0.125]], dtype=np.float32)
    x = _b(xs)
    w = np.zeros((3, 4), dtype=np.uint16)
    w[0, 3] = ONE                 # logit 0 = x[:, 3]
    w[1, 0] = ONE                 # logit 1 = x[:, 0]
    w[2, 1] = w[2, 2] = ONE       # logit 2 = x[:, 1] + x[:, 2]
    got = oracle.router_logits(x, w)
    np.testing.assert_array_equal(got, np.array([[3.0, 1.5, -1.75], [-0.125, 0.5, 3.0]],
                                                dtype=np.float32))


def test_against_numpy_float64():
    rng = np.random.default_rng(12)
    n, E, H = 64, 32, 2880
    x = _b(rng.standard_normal((n, H)))
    w = _b(rng.standard_normal((E, H)) * 0.02)
    got = oracle.router_logits(x, w, as_f32=False)
    xf, wf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(w)
    ref = xf @ wf.T
    scale = np.abs(xf) @ np.abs(wf).T
    assert np.all(np.abs(got - ref) <= 1e-13 * scale)
    f32 = oracle.router_logits(x, w)
    np.testing.assert_array_equal(f32, got.astype(np.float32))
