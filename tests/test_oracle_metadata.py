"""Pins for the oracle's routing metadata (histogram, ragged offsets, stable
expert-sorted order and its inverse, gate_scal, gather/scatter pairs).

References: numpy bincount / cumsum / stable argsort, torch.sort(stable=True)
(the exact call of the MiniMind issue, "It is removable in plain PyTorch"),
the closed form of a stable counting sort, and the permutation invariants
(gather and scatter are mutual inverses)."""
import numpy as np
import pytest
import torch

import oracle
import moe_inputs as I

CASES = [(n, E, k) for n in (1, 33, 512, 4096) for (E, k) in ((32, 4), (128, 4))] + [
    (0, 8, 2), (5, 1, 1), (100, 3, 3), (257, 16, 1)]


def _meta(n, E, k, seed=0, tie_heavy=False):
    logits = I.route_logits(n, E, seed=seed, tie_heavy=tie_heavy)
    indx, vals = oracle.route(logits, k)
    return indx, vals, oracle.metadata(indx, vals, E)


@pytest.mark.parametrize("n,E,k", CASES)
def test_against_library_routines(n, E, k):
    indx, vals, m = _meta(n, E, k)
    flat = indx.ravel()
    np.testing.assert_array_equal(m["col_sum"], np.bincount(flat, minlength=E))
    assert m["col_sum"].sum() == n * k
    np.testing.assert_array_equal(m["offs"], np.concatenate([[0], np.cumsum(m["col_sum"])]))
    np.testing.assert_array_equal(m["col_sorted"], np.argsort(flat, kind="stable"))
    t_sorted = torch.sort(torch.from_numpy(flat.astype(np.int64)), stable=True)
    np.testing.assert_array_equal(m["col_sorted"], t_sorted.indices.numpy())
    np.testing.assert_array_equal(m["gate_scal"], vals.ravel()[m["col_sorted"]])


@pytest.mark.parametrize("n,E,k", CASES)
def test_permutation_invariants(n, E, k):
    indx, _, m = _meta(n, E, k, seed=1, tie_heavy=True)
    N = n * k
    cs, rs = m["col_sorted"], m["row_sorted"]
    np.testing.assert_array_equal(np.sort(cs), np.arange(N))
    np.testing.assert_array_equal(rs[cs], np.arange(N))   # scatter after gather = id
    np.testing.assert_array_equal(cs[rs], np.arange(N))   # gather after scatter = id
    flat = indx.ravel()
    for e in range(E):
        seg = cs[m["offs"][e]:m["offs"][e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                   # stable: slot order kept
    # aliases of the first report's GatherIndx / ScatterIndx
    assert m["gather_src"] is cs and m["gather_dst"] is rs
    assert m["scatter_src"] is rs and m["scatter_dst"] is cs


def test_closed_form_position_by_brute_force():
    indx, _, m = _meta(40, 6, 3, seed=4)
    flat = indx.ravel()
    for f in range(flat.size):
        e = flat[f]
        p = m["offs"][e] + int(np.sum(flat[:f] == e))
        assert m["row_sorted"][f] == p


def test_token_ids_match_the_minimind_dispatch():
    # tok = order // k in "It is removable in plain PyTorch"
    indx, _, m = _meta(64, 8, 2, seed=5)
    order = torch.sort(torch.from_numpy(indx.ravel().astype(np.int64)), stable=True).indices
    np.testing.assert_array_equal(m["col_sorted"] // 2, (order // 2).numpy())


def test_empty_experts_and_skew():
    case = I.SKEWED.with_n(2048)
    logits = I.layer_logits(case)
    indx, vals = oracle.route(logits, case.k)
    m = oracle.metadata(indx, vals, case.E)
    assert (m["col_sum"] == 0).sum() > 10                 # many empty experts
    empty = np.nonzero(m["col_sum"] == 0)[0]
    np.testing.assert_array_equal(m["offs"][empty], m["offs"][empty + 1])
    np.testing.assert_array_equal(m["col_sorted"], np.argsort(indx.ravel(), kind="stable"))


def test_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.metadata(np.array([[0, 4]], dtype=np.int32), np.zeros((1, 2), np.uint16), 4)
