"""Pins of the oracle's accept-test variants (CPU only): the calibration
factor gamma of u < min(1, gamma p/q) and the log-space clamped test.

They are pinned by properties the definitions force, not by retyping them:
gamma = 1 is the plain test; acceptance grows with gamma (each node's test is
monotone in gamma, so the deepest fully accepted node can only get deeper);
an enormous gamma accepts every node whose p~ is positive; a tighter clamp
never accepts less; without the clamp biting, the log-space test decides as
the ratio test except within rounding of the boundary u = p/q; a gamma that
is not a positive finite number marks the tree as malformed."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl


def _case(num, **over):
    return wl.make_case(wl.config(num, **over), parts=("accept",), kind="probs")


CASES = [(1, {}), (2, dict(vocab=3000)), (3, dict(batch=6, vocab=2000, n=(10, 30)))]


@pytest.mark.parametrize("num, over", CASES)
def test_gamma_one_is_the_plain_test(num, over):
    case = _case(num, **over)
    a = oracle.accept(case)
    b = oracle.accept(case, gamma=np.ones(case["batch"], np.float32))
    for k in ("accepted_len", "path", "bonus_token", "status"):
        assert np.array_equal(a[k], b[k])


@pytest.mark.parametrize("num, over", CASES)
def test_acceptance_grows_with_gamma(num, over):
    case = _case(num, **over)
    B = case["batch"]
    lens = [oracle.accept(case, gamma=np.full(B, g, np.float32))["accepted_len"]
            for g in (0.25, 0.5, 1.0, 2.0, 4.0, 1e30)]
    for lo, hi in zip(lens, lens[1:]):
        assert np.all(lo <= hi)
    # gamma = 1e30: every node with p~ > 0 passes, so the deepest node whose
    # whole path has positive target probability is reached
    out = oracle.accept(case, gamma=np.full(B, 1e30, np.float32))
    off, par = case["node_offsets"], case["parent"]
    for b in range(B):
        n0, N = off[b], off[b + 1] - off[b]
        pq = oracle.accept(case)["pq"]
        depth = np.zeros(N, int)
        ok = np.ones(N, bool)
        for i in range(1, N):
            depth[i] = depth[par[n0 + i]] + 1
            ok[i] = ok[par[n0 + i]] and pq[n0 + i, 0] > 0
        assert out["accepted_len"][b] == depth[ok].max()


@pytest.mark.parametrize("num, over", CASES)
def test_tighter_clamp_never_accepts_less(num, over):
    case = _case(num, **over)
    l20 = oracle.accept(case, test=1, log_clamp=20.0)["accepted_len"]
    l2 = oracle.accept(case, test=1, log_clamp=2.0)["accepted_len"]
    l0 = oracle.accept(case, test=1, log_clamp=1e-3)["accepted_len"]
    assert np.all(l20 <= l2) and np.all(l2 <= l0)


@pytest.mark.parametrize("num, over", CASES)
def test_log_test_matches_ratio_test_away_from_the_boundary(num, over):
    case = _case(num, **over)
    ratio = oracle.accept(case)
    logt = oracle.accept(case, test=1, log_clamp=80.0)
    pq = ratio["pq"]
    u = case["uniforms"].astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        near = np.abs(u - pq[:, 0].astype(np.float64) / pq[:, 1]) < 1e-5
    off = case["node_offsets"]
    for b in range(case["batch"]):
        if not near[off[b] + 1: off[b + 1]].any():
            assert ratio["accepted_len"][b] == logt["accepted_len"][b]
            assert np.array_equal(ratio["path"][b], logt["path"][b])


@pytest.mark.parametrize("g", [0.0, -1.0, np.nan, np.inf])
def test_bad_gamma_marks_the_tree(g):
    case = _case(3, batch=3, vocab=500, n=(5, 9))
    gamma = np.ones(3, np.float32)
    gamma[1] = g
    out = oracle.accept(case, gamma=gamma)
    assert list(out["status"]) == [0, 5, 0] and out["accepted_len"][1] == -1
