"""Pins of the oracle's retained set (the cumulative-mass truncation that
feeds the accept pass's pruning renormalisation), CPU only.

The set is characterised without the oracle's sort: it is closed upwards in
the order (draft probability desc, token id asc); its exact 2^-40 fixed-point
mass reaches T = floor(mass * 2^40) unless it is the whole row; dropping its
last member in that order falls below T.  A uniform row has a closed form,
and on realistic rows the set agrees with the fp64 cumulative-sum recipe used
to prepare the multimodal workload's masks."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl


def _key(x):
    return np.float32(x) if (x > 0) else np.float32(0.0)  # NaN and negatives -> 0


def _check_properties(q, mass, mask_words, zf, kept):
    V = q.shape[0]
    inset = wl.unpack_mask(mask_words, V)
    T = oracle.retained_threshold(mass)
    rank = sorted(range(V), key=lambda v: (-float(_key(q[v])), v))
    pos = np.empty(V, np.int64)
    pos[rank] = np.arange(V)
    # closed upwards: the set is a prefix of the order
    assert inset.sum() == kept
    assert np.all(inset[rank[:kept]]) and not np.any(inset[rank[kept:]])
    total = sum(oracle.quantise(float(_key(q[v]))) for v in rank[:kept])
    assert total == int(zf)
    if kept < V:
        assert total >= T
    else:
        assert total >= T or sum(oracle.quantise(float(_key(x))) for x in q) < T
    if kept > 1:
        assert total - oracle.quantise(float(_key(q[rank[kept - 1]]))) < T


@pytest.mark.parametrize("seed", range(40))
def test_small_rows_satisfy_the_definition(seed):
    g = np.random.default_rng(seed)
    V = int(g.integers(1, 12))
    q = g.choice([0.0, 0.05, 0.1, 0.2, 0.3], size=V).astype(np.float32)  # many ties
    if seed % 5 == 0:
        q[g.integers(0, V)] = np.nan
    mass = float(g.choice([0.05, 0.3, 0.7, 1.0]))
    m, zf, z, kept = oracle.retained_set(q, mass)
    _check_properties(q, mass, m[0], zf[0], int(kept[0]))
    assert z[0] == np.float32(float(zf[0])) * np.float32(2.0 ** -40)


def test_uniform_row_closed_form():
    V = 1000
    q = np.full(V, np.float32(1.0 / V), np.float32)
    w = oracle.quantise(float(q[0]))
    m, zf, z, kept = oracle.retained_set(q, 0.7)
    T = oracle.retained_threshold(0.7)
    want = -(-T // w)  # ceil(T / w)
    assert kept[0] == want and zf[0] == want * w
    # ties go to the lower ids: exactly the first `want` tokens
    assert np.array_equal(wl.unpack_mask(m[0], V), np.arange(V) < want)


def test_zero_and_tiny_rows_keep_everything():
    for q in (np.zeros(70, np.float32), np.full(70, np.float32(1e-13), np.float32)):
        m, zf, z, kept = oracle.retained_set(q, 0.7)
        assert kept[0] == 70 and wl.unpack_mask(m[0], 70).all()


@pytest.mark.parametrize("num", [2, 4])
def test_agrees_with_the_fp64_recipe_on_softmax_rows(num):
    case = wl.make_case(wl.config(num, batch=1, n=(6, 6), depth=2), parts=("accept",))
    rows = case["draft_probs"][:4]
    m, zf, z, kept = oracle.retained_set(rows, 0.7)
    for r in range(rows.shape[0]):
        assert np.array_equal(m[r], wl.retained_mask_row(rows[r], 0.7)), r
        _check_properties(rows[r], 0.7, m[r], zf[r], int(kept[r]))
