"""Pins for the oracle's router top-k and gate weights.

Top-k order (logit descending, ties to the lower expert id) is checked
against brute force over every ordered k-subset, numpy's argmax (first
maximum) and numpy's stable argsort; gate weights against closed forms and
a numpy float64 softmax."""
import itertools
import math

import numpy as np
import pytest

import oracle
import moe_inputs as I


def _brute_topk(row: np.ndarray, k: int):
    """Largest sequence of (logit, -expert) keys over all ordered k-subsets."""
    best, best_key = None, None
    for perm in itertools.permutations(range(row.size), k):
        key = tuple((float(row[e]), -e) for e in perm)
        if best_key is None or key > best_key:
            best, best_key = perm, key
    return list(best)


@pytest.mark.parametrize("E", [1, 2, 3, 5, 6])
@pytest.mark.parametrize("source", ["normal", "ints", "bf16"])
def test_topk_matches_brute_force(E, source):
    n = 24
    if source == "normal":
        logits = I.route_logits(n, E, seed=E)
    elif source == "ints":
        logits = I.small_int_logits(n, E, seed=E, levels=1)
    else:
        logits = I.route_logits(n, E, seed=E, tie_heavy=True)
    for k in range(1, E + 1):
        indx, _ = oracle.route(logits, k)
        for t in range(n):
            assert list(indx[t]) == _brute_topk(logits[t], k), (t, k, logits[t])


@pytest.mark.parametrize("n,E", [(512, 32), (300, 128), (64, 256)])
def test_top1_is_first_argmax(n, E):
    for logits in (I.route_logits(n, E), I.small_int_logits(n, E, levels=2)):
        indx, _ = oracle.route(logits, 1)
        np.testing.assert_array_equal(indx[:, 0], np.argmax(logits, axis=1))


@pytest.mark.parametrize("E", [4, 16, 33])
def test_topE_is_stable_descending_argsort(E):
    for logits in (I.route_logits(50, E), I.small_int_logits(50, E, levels=2)):
        indx, _ = oracle.route(logits, E)
        np.testing.assert_array_equal(indx, np.argsort(-logits, axis=1, kind="stable"))


def test_signed_zero_is_a_tie():
    logits = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]], dtype=np.float32)
    indx, _ = oracle.route(logits, 2)
    assert indx.tolist() == [[0, 1], [0, 1]]


def test_nonfinite_logits_rejected():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0.0, np.nan]], dtype=np.float32), 1)


def _bf16(v: float) -> int:
    return int(oracle.f64_to_bf16(np.array([v]))[0])


def test_gate_closed_forms():
    # softmax over the k selected with k = 1 is exactly 1
    _, v = oracle.route(I.route_logits(40, 8), 1, "softmax_topk")
    assert (v == 0x3F80).all()
    # two equal selected logits -> 1/2 each
    _, v = oracle.route(np.array([[3.0, 3.0, -1.0]], dtype=np.float32), 2, "softmax_topk")
    assert v.tolist() == [[0x3F00, 0x3F00]]
    # softmax over all E equal logits -> 1/E
    for E, expected in ((4, 0x3E80), (3, _bf16(1.0 / 3.0))):
        _, v = oracle.route(np.zeros((2, E), dtype=np.float32), 1, "softmax_all")
        assert (v == expected).all(), (E, v)
    assert _bf16(1.0 / 3.0) == 0x3EAB  # 171/512, worked by hand
    # logits that differ by exactly log(3) in float64 terms: weights 3/4, 1/4
    l1 = np.float32(0.5)
    l0 = np.float32(np.float64(l1) + math.log(3.0))
    w0 = 1.0 / (1.0 + math.exp(float(l1) - float(l0)))
    _, v = oracle.route(np.array([[l0, l1]], dtype=np.float32), 2, "softmax_topk")
    assert v.tolist() == [[_bf16(w0), _bf16(1.0 - w0)]]
    assert abs(w0 - 0.75) < 1e-7


def _softmax64(l: np.ndarray) -> np.ndarray:
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def _assert_correctly_rounded(bits: np.ndarray, exact: np.ndarray):
    """bits must be the bf16 nearest to `exact` (slack 1e-9 relative for the
    different float64 summation order)."""
    got = oracle.bf16_to_f64(bits)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    assert np.all(np.abs(got - exact) <= 0.5 * ulp * (1 + 1e-9)), np.max(np.abs(got - exact) / ulp)


@pytest.mark.parametrize("E,k", [(8, 2), (32, 4), (128, 4), (16, 1)])
def test_gate_values_against_numpy_softmax(E, k):
    logits = I.route_logits(200, E, seed=7)
    indx, v_topk = oracle.route(logits, k, "softmax_topk")
    sel = np.take_along_axis(logits.astype(np.float64), indx, axis=1)
    _assert_correctly_rounded(v_topk, _softmax64(sel))
    indx2, v_all = oracle.route(logits, k, "softmax_all")
    np.testing.assert_array_equal(indx, indx2)
    p = _softmax64(logits.astype(np.float64))
    _assert_correctly_rounded(v_all, np.take_along_axis(p, indx, axis=1))
    # the selected weights sum to 1 (within k roundings)
    assert np.all(np.abs(oracle.bf16_to_f64(v_topk).sum(1) - 1.0) <= k * 2.0 ** -8)


def test_all_and_topk_agree_when_k_is_E():
    logits = I.route_logits(100, 6, seed=3)
    _, a = oracle.route(logits, 6, "softmax_all")
    _, b = oracle.route(logits, 6, "softmax_topk")
    d = np.abs(a.astype(np.int32) - b.astype(np.int32))
    assert d.max() <= 1 and (d == 0).mean() > 0.99
