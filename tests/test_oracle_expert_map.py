"""Pins of the oracle's expert map (expert parallelism: a rank holds a subset
of the experts; a slot whose expert lives on another rank is marked -1 and
dropped). "Reuse topk SparseMatrix routing metadata in GPT-OSS MoE forward",
功能与动机 (expert-parallel routing) and 风险与影响 (the -1 slots).

The mapped oracle is pinned against the unmapped one (itself pinned by the
other oracle tests) and against numpy: the identity map changes nothing; the
metadata of a partition is the stable sort of the kept slots; every kept
slot's gate-weighted expert output is the full layer's, bit for bit; and the
ranks' outputs add up to the full layer's (exactly at k = 1)."""
import numpy as np
import pytest

import oracle
import moe_inputs as I

E, H, I_ = 8, 64, 128


def _layer(n, k, seed=3, act="swiglu", layout="packed"):
    c = I.LayerCase("emap", n=n, H=H, E=E, k=k, I=I_, act=act, layout=layout, w_std=0.05,
                    seed=seed)
    h = I.layer_inputs(c)
    indx, vals = oracle.route(h["logits"], k, c.gating)
    return c, h, indx, vals


def _rank_map(ranks, r, order=None):
    """Experts split into `ranks` contiguous blocks; rank r's local ids
    (optionally permuted by `order`)."""
    m = np.full(E, -1, dtype=np.int32)
    mine = np.arange(E)[np.arange(E) * ranks // E == r]
    loc = np.arange(mine.size) if order is None else np.asarray(order)
    m[mine] = loc
    return m, mine


def _local_weights(h, mine, m):
    inv = np.empty(mine.size, dtype=np.int64)
    inv[m[mine]] = mine  # local id -> global expert
    return h["w13"][inv], h["w2"][inv]


def _numpy_metadata(indx, vals, m, n_local):
    loc = m[indx.ravel()]
    kept = np.flatnonzero(loc >= 0)
    col_sum = np.bincount(loc[kept], minlength=n_local)
    col_sorted = kept[np.argsort(loc[kept], kind="stable")]
    row_sorted = np.full(indx.size, -1, dtype=np.int64)
    row_sorted[col_sorted] = np.arange(col_sorted.size)
    return col_sum, col_sorted, row_sorted, vals.ravel()[col_sorted]


def test_identity_map_changes_nothing():
    c, h, indx, vals = _layer(40, 2)
    ident = np.arange(E, dtype=np.int32)
    a = oracle.metadata(indx, vals, E)
    b = oracle.metadata(indx, vals, E, expert_map=ident, n_local=E)
    for key in ("col_sum", "offs", "col_sorted", "row_sorted", "gate_scal"):
        np.testing.assert_array_equal(a[key], b[key])
    kw = dict(act=c.act, layout=c.layout)
    out = oracle.ffn(h["x"], indx, vals, h["w13"], h["w2"], **kw)
    out_m = oracle.ffn(h["x"], indx, vals, h["w13"], h["w2"], expert_map=ident, n_experts=E, **kw)
    np.testing.assert_array_equal(out, out_m)


@pytest.mark.parametrize("ranks,k", [(2, 2), (4, 3), (8, 1)])
def test_partition_metadata_is_the_stable_sort_of_the_kept_slots(ranks, k):
    c, h, indx, vals = _layer(57, k)
    seen = np.zeros(indx.size, dtype=np.int64)
    for r in range(ranks):
        m, mine = _rank_map(ranks, r)
        md = oracle.metadata(indx, vals, E, expert_map=m, n_local=mine.size)
        col_sum, col_sorted, row_sorted, gate = _numpy_metadata(indx, vals, m, mine.size)
        np.testing.assert_array_equal(md["col_sum"], col_sum)
        np.testing.assert_array_equal(md["offs"], np.concatenate([[0], np.cumsum(col_sum)]))
        np.testing.assert_array_equal(md["col_sorted"], col_sorted)
        np.testing.assert_array_equal(md["row_sorted"], row_sorted)
        np.testing.assert_array_equal(md["gate_scal"], gate)
        seen[md["col_sorted"]] += 1
    np.testing.assert_array_equal(seen, 1)  # every slot is kept by exactly one rank


@pytest.mark.parametrize("order", [None, [2, 0, 3, 1]])
def test_kept_slots_compute_the_full_layers_expert_outputs(order):
    """Rank 1 of 2 (experts 4..7, local ids in `order`): each kept slot's
    gate-weighted expert output and intermediate equal the unmapped layer's
    bit for bit (so local ids index the local weights correctly); dropped
    slots are zero."""
    c, h, indx, vals = _layer(33, 2, act="swiglu_oai", layout="interleaved")
    kw = dict(act=c.act, layout=c.layout)
    _, y_full, h_full = oracle.ffn(h["x"], indx, vals, h["w13"], h["w2"], want_slots=True, **kw)
    m, mine = _rank_map(2, 1, order)
    w13_l, w2_l = _local_weights(h, mine, m)
    _, y_r, h_r = oracle.ffn(h["x"], indx, vals, w13_l, w2_l, want_slots=True, expert_map=m,
                             n_experts=E, **kw)
    kept = m[indx] >= 0
    assert kept.any() and (~kept).any()
    np.testing.assert_array_equal(y_r[kept], y_full[kept])
    np.testing.assert_array_equal(h_r[kept], h_full[kept])
    assert not y_r[~kept].any() and not h_r[~kept].any()


def test_ranks_add_up_to_the_full_layer():
    """k = 1: each token's one expert lives on one rank, which reproduces the
    full output row exactly; the others give zero rows. k = 3 over 4 ranks:
    the ranks' bf16 outputs add up to the full output within their roundings
    (each at most half a bf16 ulp, 2^-8 relative)."""
    c, h, indx, vals = _layer(29, 1)
    full = oracle.ffn(h["x"], indx, vals, h["w13"], h["w2"], act=c.act, layout=c.layout)
    total = np.zeros(full.shape)
    for r in range(2):
        m, mine = _rank_map(2, r)
        w13_l, w2_l = _local_weights(h, mine, m)
        out = oracle.ffn(h["x"], indx, vals, w13_l, w2_l, expert_map=m, n_experts=E, act=c.act,
                         layout=c.layout)
        mine_tok = m[indx[:, 0]] >= 0
        np.testing.assert_array_equal(out[mine_tok], full[mine_tok])
        assert not out[~mine_tok].any()
        total += oracle.bf16_to_f64(out)
    np.testing.assert_array_equal(oracle.f64_to_bf16(total), full)

    c, h, indx, vals = _layer(29, 3, seed=5)
    full = oracle.bf16_to_f64(oracle.ffn(h["x"], indx, vals, h["w13"], h["w2"], act=c.act,
                                         layout=c.layout))
    total, mag = np.zeros(full.shape), np.abs(full)
    for r in range(4):
        m, mine = _rank_map(4, r)
        w13_l, w2_l = _local_weights(h, mine, m)
        part = oracle.bf16_to_f64(oracle.ffn(h["x"], indx, vals, w13_l, w2_l, expert_map=m,
                                             n_experts=E, act=c.act, layout=c.layout))
        total += part
        mag += np.abs(part)
    assert np.all(np.abs(total - full) <= 2.0 ** -8 * mag)
    assert np.abs(full).max() > 0


def test_no_local_expert_drops_every_slot():
    c, h, indx, vals = _layer(10, 2)
    m = np.full(E, -1, dtype=np.int32)
    md = oracle.metadata(indx, vals, E, expert_map=m, n_local=1)
    np.testing.assert_array_equal(md["col_sum"], [0])
    np.testing.assert_array_equal(md["offs"], [0, 0])
    assert md["col_sorted"].size == 0 and (md["row_sorted"] == -1).all()
    out = oracle.ffn(h["x"], indx, vals, h["w13"][:1], h["w2"][:1], expert_map=m, n_experts=E,
                     act=c.act, layout=c.layout)
    assert not out.any()


@pytest.mark.parametrize("bad", [2, -2])
def test_map_entries_outside_the_local_range_are_rejected(bad):
    c, h, indx, vals = _layer(6, 2)
    m, mine = _rank_map(4, 0)  # 2 local experts
    m[5] = bad
    with pytest.raises(ValueError):
        oracle.metadata(indx, vals, E, expert_map=m, n_local=mine.size)
