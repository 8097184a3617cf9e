"""Pins of the oracle's multi-candidate accept walk (test 2; CPU only).

Siblings are tried in index order against the current target distribution,
and every rejection replaces it by its normalised residual max(0, cur - q)
(multi-step speculative sampling).  The pins do not retype the update; they
check what the definition forces:
- on a chain every node has one child, so the walk is the single-candidate
  walk: identical results to test 0, with and without a retained-set mask and
  a calibration factor;
- losslessness: when the candidate tokens are independent draws from the
  draft row q, the first emitted token (the first accepted child's token, or
  the bonus when all are rejected) is distributed as the target row p;
- hand-worked dyadic cases where every quantity is exact: targets with no
  mass on the candidates, target equal to draft, and a second sibling tested
  against the residual left by the first."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl
from test_oracle_accept_pins import accept_case, draw_index, fix40

F32 = np.float32


def _run(case, test, gamma=None):
    return oracle.accept(case, test=test, gamma=gamma)


# ---------------------------------------------------------------- chains
def random_chains(seed, n_trees, V, nmax, mask_frac=None):
    g = wl.rng(seed, 501)
    parents, T, D, toks, U = [], [], [], [], []
    for _ in range(n_trees):
        n = int(g.integers(1, nmax + 1))
        par = [-1] + list(range(n - 1))
        P = wl._softmax32(g.normal(0, 1.5, (n, V)))
        Q = wl._softmax32(np.log(np.maximum(P.astype(np.float64), 1e-30)) + g.normal(0, 0.7, (n, V)))
        qd = Q.astype(np.float64)
        tk = [-1] + [int(g.choice(V, p=qd[i - 1] / qd[i - 1].sum())) for i in range(1, n)]
        parents.append(par), T.append(P), D.append(Q), toks.extend(tk)
        U.extend((g.integers(0, 1 << 24, n) * 2.0 ** -24).astype(F32))
    mask = None
    if mask_frac is not None:
        tot = sum(len(p) for p in parents)
        W = (V + 31) // 32
        bits = g.random((tot, W * 32)) < mask_frac
        words = np.zeros((tot, W), np.uint64)
        for k in range(32):
            words |= bits[:, k::32].astype(np.uint64) << np.uint64(k)
        mask = words.astype(np.uint32)
    return accept_case(parents, V, np.concatenate(T), np.concatenate(D), toks, U, mask=mask)


@pytest.mark.parametrize("mask_frac", [None, 0.6])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chain_is_the_single_candidate_walk(seed, mask_frac):
    case = random_chains(seed, 24, 97, 9, mask_frac)
    for gamma in (None, np.full(24, 1.7, F32)):
        a, b = _run(case, 0, gamma), _run(case, 2, gamma)
        for k in ("accepted_len", "path", "bonus_token", "status"):
            assert np.array_equal(a[k], b[k]), (k, seed, mask_frac)
        # the (p~, q~) each tested node saw: every node of the accepted prefix
        # and the first rejected one carry test 0's values
        off = case["node_offsets"]
        for t in range(24):
            n = a["accepted_len"][t]
            seen = range(off[t] + 1, min(off[t] + n + 2, off[t + 1]))
            for i in seen:
                assert np.array_equal(a["pq"][i], b["pq"][i])


# ---------------------------------------------------------------- losslessness
def test_first_token_is_distributed_as_the_target():
    """Root with k candidates drawn i.i.d. from q; over many trees the first
    emitted token follows p (4-sigma bounds per token)."""
    V, k, n_trees = 6, 3, 30000
    p = np.array([0.30, 0.25, 0.20, 0.15, 0.07, 0.03], np.float64)
    q = np.array([0.05, 0.10, 0.15, 0.20, 0.25, 0.25], np.float64)
    P, Q = p.astype(F32), q.astype(F32)
    g = wl.rng(11, 502)
    toks = g.choice(V, size=(n_trees, k), p=q)
    U = (g.integers(0, 1 << 24, (n_trees, k + 1)) * 2.0 ** -24).astype(F32)
    parents = [[-1] + [0] * k for _ in range(n_trees)]
    tokens, uni = [], []
    for t in range(n_trees):
        tokens += [-1] + list(toks[t])
        uni += list(U[t])
    n = k + 1
    target = np.tile(P, (n_trees * n, 1))
    draft = np.tile(Q, (n_trees * n, 1))
    case = accept_case(parents, V, target, draft, tokens, uni)
    r = _run(case, 2)
    first = np.where(r["accepted_len"] > 0,
                     np.asarray(tokens, np.int64).reshape(n_trees, n)[np.arange(n_trees),
                                                                     np.maximum(r["path"][:, 0], 0)],
                     r["bonus_token"])
    emp = np.bincount(first, minlength=V) / n_trees
    sd = np.sqrt(p * (1 - p) / n_trees)
    assert np.all(np.abs(emp - p) <= 4 * sd + 1e-4), (emp, p)
    # and not distributed as q (the test has power)
    assert np.abs(emp - q).max() > 0.1


# ---------------------------------------------------------------- worked cases
def _star(p_rows, q_rows, child_tokens, u, u0):
    """Root 0 with the given children (all leaves); rows per node."""
    k = len(child_tokens)
    V = len(p_rows[0])
    target = np.array([p_rows[0]] + [p_rows[0]] * k, F32)
    draft = np.array([q_rows[0]] + [q_rows[0]] * k, F32)
    return accept_case([[-1] + [0] * k], V, target, draft, [-1] + list(child_tokens),
                       [u0] + list(u))


def test_no_target_mass_on_the_candidates_draws_from_the_target():
    # every candidate has p = 0: all rejected; the residual is p itself each
    # time (exact dyadic values, S = 2^40), so the bonus is a draw from p
    p = [0.5, 0.25, 0.25, 0.0, 0.0]
    q = [0.0, 0.0, 0.0, 0.5, 0.5]
    for u0 in (0.1, 0.49, 0.5, 0.74, 0.75, 0.99):
        r = _run(_star([p], [q], [3, 4, 3], [0.01, 0.5, 0.99], u0), 2)
        assert r["accepted_len"][0] == 0
        assert r["bonus_token"][0] == draw_index([fix40(x) for x in p], u0)


def test_target_equal_to_draft_accepts_the_first_child_chain():
    # p = q: u q < q for every u < 1, so the walk follows first children
    V = 8
    row = np.array([0.5, 0.125, 0.125, 0.0625, 0.0625, 0.0625, 0.0625, 0.0], F32)
    par = [-1, 0, 0, 1, 1, 3, 2]
    toks = [-1, 1, 0, 2, 3, 4, 5]
    n = len(par)
    rows = np.tile(row, (n, 1))
    case = accept_case([par], V, rows, rows, toks, [0.3] + [0.999] * (n - 1))
    r = _run(case, 2)
    assert list(r["path"][0][:3]) == [1, 3, 5] and r["accepted_len"][0] == 3
    assert r["bonus_token"][0] == draw_index([fix40(x) for x in row], F32(0.3))


@pytest.mark.parametrize("tok2, u0, want_len, want_bonus",
                         [(2, 0.5, 1, None), (0, 0.5, 1, None), (1, 0.5, 0, 0), (1, 0.9, 0, 2)])
def test_second_sibling_sees_the_residual(tok2, u0, want_len, want_bonus):
    # p = [1/2, 1/4, 1/4, 0], q = [1/4, 1/2, 1/8, 1/8].  Child 1 (token 1,
    # u = 3/4): 3/8 < 1/4 fails.  Residual max(0, p - q) = [1/4, 0, 1/8, 0],
    # S = 3/8 exactly, cur = [2/3, 0, 1/3, 0] (rounded).  Child 2 with token 2
    # or 0 passes (u q <= 1/4 < cur); with token 1 (cur = 0) it fails, and the
    # bonus comes from max(0, cur - q) = [~0.4167, 0, ~0.2083, 0], i.e. 2:1
    # between tokens 0 and 2.
    p = [0.5, 0.25, 0.25, 0.0]
    q = [0.25, 0.5, 0.125, 0.125]
    r = _run(_star([p], [q], [1, tok2], [0.75, 0.999], u0), 2)
    assert r["accepted_len"][0] == want_len
    if want_len == 1:
        assert r["path"][0][0] == 2
        # the accepted child is a leaf: its bonus is a draw from p (its row)
        assert r["bonus_token"][0] == draw_index([fix40(x) for x in p], F32(u0))
    else:
        assert r["bonus_token"][0] == want_bonus
    # the first test saw p~(1) = 1/4; the second the residual value
    assert r["pq"][1][0] == F32(0.25)
    cur = {2: Fraction(1, 3), 0: Fraction(2, 3), 1: Fraction(0)}[tok2]
    assert abs(Fraction(float(r["pq"][2][0])) - cur) < Fraction(1, 1 << 22)
