"""Pins of the accept oracle against what the pages and mathematics fix.

* The per-node test u < min(1, p_target/p_draft) with parallel uniforms, the
  root-first walk cut at the first rejection and the longest accepted path
  (edge-cloud tree-attention page, §2.2.3).
* A chain tree is standard speculative decoding (on-device LLM pruning page
  §1.2: draft, one verification pass, accept/reject with resampling at the
  rejection) -> a separately written textbook loop.
* Brute force over all root-to-node paths of every small tree.
* Importance correction (on-device LLM pruning page §2.2.1-§2.2.2, §7.1):
  q~ = q * 1_R / Z; pruned tokens can never be accepted nor drawn.
* Losslessness (the pages' "lossless" claim; Leviathan et al. 2023): chains
  whose draft token is drawn from q emit a first token distributed as p, and
  the first-node acceptance rate is sum_x min(p, q) (alpha of §7.1 of the
  edge-cloud page).
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def accept_case(parents, V, target, draft, tokens, uniforms, mask=None, kind="probs",
                max_nodes=None):
    ns = [len(p) for p in parents]
    off = np.zeros(len(parents) + 1, np.int32)
    off[1:] = np.cumsum(ns)
    return dict(node_offsets=off, parent=np.concatenate([np.asarray(p, np.int32) for p in parents]),
                vocab=V, target=np.asarray(target, F32), draft_probs=np.asarray(draft, F32),
                draft_tokens=np.asarray(tokens, np.int32), uniforms=np.asarray(uniforms, F32),
                retained_mask=mask, kind=kind, max_nodes=max_nodes or max(ns))


# ---------------------------------------------------------------- fixed point
def fix40(r):
    """floor(clamp(r, 0, 32) * 2^40) by exact rational arithmetic."""
    r = F32(r)
    if not (r > 0):
        return 0
    r = min(Fraction(float(r)), Fraction(32))
    return int(r * 2 ** 40)


def draw_index(weights_fix, u):
    S = sum(weights_fix)
    t = int(Fraction(float(F32(u))) * S)  # floor for non-negative values
    cum = 0
    for v, f in enumerate(weights_fix):
        cum += f
        if cum > t:
            return v
    return None


def int_to_f32_rn(n: int) -> float:
    """Nearest-even fp32 of a non-negative integer, by integer arithmetic."""
    if n == 0:
        return 0.0
    e = n.bit_length()
    if e <= 24:
        return float(n)
    sh = e - 24
    m, rem = n >> sh, n & ((1 << sh) - 1)
    half = 1 << (sh - 1)
    if rem > half or (rem == half and (m & 1)):
        m += 1
    return float(m << sh)


def test_quantise_and_draw_exact_against_big_integers():
    g = wl.rng(1, 1)
    rs = np.concatenate([g.random(2000).astype(F32), F32([0, 1, 2 ** -40, 2 ** -41, 31.99, 32,
                                                          40, np.nan, -1, 3e-13])])
    for r in rs:
        assert oracle.quantise(float(r)) == fix40(r)
    for _ in range(2000):
        u = F32(int(g.integers(0, 1 << 24)) * 2.0 ** -24)
        S = int(g.integers(1, 1 << 63))
        assert oracle.scaled_draw(float(u), S) == int(Fraction(float(u)) * S)
    assert oracle.scaled_draw(float(F32(1 - 2 ** -24)), (1 << 64) - 1) == \
        int(Fraction(float(F32(1 - 2 ** -24))) * ((1 << 64) - 1))


# ------------------------------------------------------------ textbook chain
def textbook_chain(P, Q, tokens, u):
    """Standard speculative decoding on one chain: rows P[j], Q[j] are the
    target/draft distributions after token j; tokens[1:] are the drafts."""
    n = len(tokens)
    k = 0
    while k + 1 < n:
        i = k + 1
        x = tokens[i]
        if F32(u[i]) * F32(Q[k][x]) < F32(P[k][x]):
            k = i
        else:
            break
    if k + 1 < n:  # rejected after k accepted tokens: residual at row k
        w = [fix40(F32(P[k][v]) - F32(Q[k][v])) for v in range(len(P[k]))]
        if sum(w) == 0:
            w = [fix40(P[k][v]) for v in range(len(P[k]))]
    else:          # every draft accepted: sample the next token from p
        w = [fix40(P[k][v]) for v in range(len(P[k]))]
    return k, draw_index(w, u[0])


@pytest.mark.parametrize("seed", range(6))
def test_chain_matches_textbook_speculative_decoding(seed):
    g = wl.rng(seed, 3)
    V = 24
    parents, T, D, toks, U, exp = [], [], [], [], [], []
    for b in range(40):
        n = int(g.integers(1, 9))
        P = wl._softmax32(g.normal(0, 1.5, (n, V)))
        Q = wl._softmax32(g.normal(0, 1.5, (n, V)))
        qn = Q.astype(np.float64)
        qn /= qn.sum(axis=1, keepdims=True)
        tk = [-1] + [int(g.choice(V, p=qn[i - 1])) for i in range(1, n)]
        u = (g.integers(0, 1 << 24, n) * 2.0 ** -24).astype(F32)
        parents.append([-1] + list(range(n - 1)))
        T.append(P), D.append(Q), toks.extend(tk), U.extend(u)
        exp.append(textbook_chain(P, Q, tk, u))
    case = accept_case(parents, V, np.concatenate(T), np.concatenate(D), toks, U, max_nodes=8)
    out = oracle.accept(case)
    for b, (k, tok) in enumerate(exp):
        assert out["status"][b] == 0
        assert out["accepted_len"][b] == k
        assert list(out["path"][b, :k]) == list(range(1, k + 1))
        assert np.all(out["path"][b, k:] == -1)
        assert out["bonus_token"][b] == tok


# ------------------------------------------------------- brute force on trees
def all_trees(n):
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1] + list(choice)


def brute_force_longest(par, acc):
    best = (0, 0)  # (depth, -index) maximised
    best_node = 0
    for i in range(1, len(par)):
        path, k = [], i
        while k > 0:
            path.append(k)
            k = par[k]
        if all(acc[j] for j in path):
            key = (len(path), -i)
            if key > best:
                best, best_node = key, i
    path, k = [], best_node
    while k > 0:
        path.append(k)
        k = par[k]
    return best[0], path[::-1]


def test_walk_brute_force_all_trees_up_to_7_nodes():
    """Every tree with <= 7 nodes and random accept patterns: the deepest node
    whose whole root path is accepted, ties to the smallest index."""
    g = wl.rng(7, 7)
    V = 8
    parents, T, D, toks, U, want = [], [], [], [], [], []
    for n in range(1, 8):
        for par in all_trees(n):
            for _ in range(2 if n < 7 else 1):
                acc = [False] + [bool(g.integers(0, 2)) for _ in range(1, n)]
                P = np.full((n, V), 0.01, F32)
                Q = np.full((n, V), 0.01, F32)
                tk = [-1]
                for i in range(1, n):
                    x = i  # distinct among siblings
                    tk.append(x)
                    # accepted: u*q = 0.5*0.25 < 0.5 ; rejected: 0.5*0.5 = 0.25 !< 0.1
                    P[par[i], x], Q[par[i], x] = (0.5, 0.25) if acc[i] else (0.1, 0.5)
                parents.append(par), T.append(P), D.append(Q), toks.extend(tk)
                U.extend([0.3] + [0.5] * (n - 1))
                want.append(brute_force_longest(par, acc))
    case = accept_case(parents, V, np.concatenate(T), np.concatenate(D), toks, U, max_nodes=7)
    out = oracle.accept(case)
    for b, (ln, path) in enumerate(want):
        assert out["accepted_len"][b] == ln
        assert list(out["path"][b, :ln]) == path


# ------------------------------------------------------------------ specials
def _one(p_vals, q_vals, u, V=4, x=2):
    P = np.zeros((2, V), F32)
    Q = np.zeros((2, V), F32)
    P[0, x], Q[0, x] = p_vals, q_vals
    P[0, (x + 1) % V] = 1.0 - P[0, x] if np.isfinite(P[0, x]) else 0.5
    P[1, 0] = 1.0
    case = accept_case([[-1, 0]], V, P, Q, [-1, x], [0.25, u])
    return oracle.accept(case)


def test_acceptance_special_values():
    assert _one(0.3, 0.0, 0.9)["accepted_len"][0] == 1   # q = 0, p > 0: accept
    assert _one(0.0, 0.0, 0.0)["accepted_len"][0] == 0   # p = 0: reject, even u = 0
    assert _one(0.0, 0.5, 0.1)["accepted_len"][0] == 0
    assert _one(0.2, 0.7, 0.0)["accepted_len"][0] == 1   # u = 0, p > 0: accept
    assert _one(np.nan, 0.5, 0.1)["accepted_len"][0] == 0  # NaN rejects
    # strictness: u*q == p rejects
    assert _one(0.25, 0.5, 0.5)["accepted_len"][0] == 0
    assert _one(np.nextafter(F32(0.25), F32(1)), 0.5, 0.5)["accepted_len"][0] == 1


def test_root_only_tree_draws_from_p():
    V = 8
    P = np.zeros((1, V), F32)
    P[0, :] = 0.125  # uniform over 8 tokens: token k exactly on [k/8, (k+1)/8)
    for k in range(8):
        for u, want in ((k / 8, k), (k / 8 + 2 ** -24, k), (k / 8 - 2 ** -24, k - 1)):
            if u < 0:
                continue
            out = oracle.accept(accept_case([[-1]], V, P, P * 0, [-1], [u]))
            assert out["accepted_len"][0] == 0 and out["bonus_token"][0] == want


def test_one_hot_residual_always_draws_that_token():
    V = 16
    P = np.zeros((2, V), F32)
    Q = np.zeros((2, V), F32)
    P[0, 3], P[0, 9] = 0.5, 0.5
    Q[0, 3] = 0.75
    Q[0, 9] = 0.25  # residual = 0.25 at token 9 only
    Q[0, 3] = 0.75
    for u0 in np.linspace(0, 1 - 2 ** -24, 17):
        # draft token 3 rejected with u = 0.9 (0.9*0.75 > 0.5)
        out = oracle.accept(accept_case([[-1, 0]], V, P, Q, [-1, 3], [u0, 0.9]))
        assert out["accepted_len"][0] == 0 and out["bonus_token"][0] == 9


def test_all_zero_mass_falls_back_to_argmax():
    V = 8
    P = np.zeros((1, V), F32)
    P[0, 5] = 1e-13  # below the 2^-40 quantum
    P[0, 6] = 1e-13
    out = oracle.accept(accept_case([[-1]], V, P, P, [-1], [0.7]))
    assert out["bonus_token"][0] == 5


def test_malformed_trees_report_status():
    V = 4
    P = np.full((3, V), 0.25, F32)
    for par, toks in (([0, 0, 1], [-1, 1, 2]), ([-1, 1, 0], [-1, 1, 2]), ([-1, 0, 0], [-1, 1, 4])):
        out = oracle.accept(accept_case([par], V, P, P, toks, [0.5] * 3))
        assert out["status"][0] == 5 and out["accepted_len"][0] == -1
        assert out["bonus_token"][0] == -1 and np.all(out["path"][0] == -1)


# ---------------------------------------------------------------- renorm
def _rand_mask(g, V, keep_frac):
    kept = g.random(V) < keep_frac
    words = np.zeros((V + 31) // 32, np.uint32)
    for v in np.nonzero(kept)[0]:
        words[v // 32] |= np.uint32(1 << (v % 32))
    return words, kept


def test_retained_mass_is_exact_fixed_point_sum():
    g = wl.rng(3, 3)
    for V in (1, 31, 32, 33, 1000):
        q = wl._softmax32(g.normal(0, 2, (1, V)))[0]
        words, kept = _rand_mask(g, V, 0.4)
        S = sum(fix40(q[v]) for v in range(V) if kept[v])
        want = F32(int_to_f32_rn(S) * 2.0 ** -40)
        assert oracle.retained_mass(q, words) == want
        S_all = sum(fix40(x) for x in q)
        assert oracle.retained_mass(q, None) == F32(int_to_f32_rn(S_all) * 2.0 ** -40)


def test_pruned_tokens_never_accepted_nor_drawn():
    g = wl.rng(5, 5)
    V, n_trees = 40, 60
    parents, T, D, toks, U, masks, keptsets = [], [], [], [], [], [], []
    for b in range(n_trees):
        n = int(g.integers(1, 7))
        par = [-1] + [int(g.integers(0, i)) for i in range(1, n)]
        P = wl._softmax32(g.normal(0, 1, (n, V)))
        Q = wl._softmax32(g.normal(0, 1, (n, V)))
        mk = [_rand_mask(g, V, 0.5) for _ in range(n)]
        tk = [-1] + [int(g.integers(0, V)) for _ in range(1, n)]
        parents.append(par), T.append(P), D.append(Q), toks.extend(tk)
        U.extend((g.integers(0, 1 << 24, n) * 2.0 ** -24).astype(F32))
        masks.extend([m[0] for m in mk])
        keptsets.append([m[1] for m in mk])
    case = accept_case(parents, V, np.concatenate(T), np.concatenate(D), toks, U,
                       mask=np.stack(masks), max_nodes=6)
    out = oracle.accept(case)
    off = case["node_offsets"]
    for b in range(n_trees):
        par = parents[b]
        for i in out["path"][b, : out["accepted_len"][b]]:
            assert keptsets[b][par[i]][toks[off[b] + i]]
        cut = out["path"][b, out["accepted_len"][b] - 1] if out["accepted_len"][b] else 0
        if keptsets[b][cut].any():
            assert keptsets[b][cut][out["bonus_token"][b]]
        # p~/q~ of every tested node: p/Z, q/Z on R; 0 off R
        for i in range(1, len(par)):
            j, x = par[i], toks[off[b] + i]
            ptq = out["pq"][off[b] + i]
            if keptsets[b][j][x]:
                Z = F32(oracle.retained_mass(D[b][j], masks[off[b] + j]))
                assert ptq[0] == F32(T[b][j][x]) / Z and ptq[1] == F32(D[b][j][x]) / Z
            else:
                assert ptq[0] == 0 and ptq[1] == 0


def test_all_ones_mask_matches_no_mask_up_to_near_ties():
    c = wl.make_case(wl.config(3, batch=6, vocab=257, prefix=(16, 16)), parts=("accept",))
    V = c["vocab"]
    ones = np.full((c["total_nodes"], (V + 31) // 32), 0xFFFFFFFF, np.uint32)
    a = oracle.accept(c)
    cm = dict(c)
    cm["retained_mask"] = ones
    m = oracle.accept(cm)
    # Z is 1 up to 2^-40 quanta, so the test u*q~ < p~ can only flip at near-ties
    diff = np.nonzero(a["accepted_len"] != m["accepted_len"])[0]
    for b in diff:
        off = c["node_offsets"]
        u = c["uniforms"][off[b]:off[b + 1]]
        pq = a["pq"][off[b]:off[b + 1]]
        gap = np.abs(u[1:] * pq[1:, 1] - pq[1:, 0]) / np.maximum(pq[1:, 0], 1e-30)
        assert gap.min() < 1e-5
    assert len(diff) <= 1


# ---------------------------------------------------------------- logits mode
def test_logits_mode_equals_probs_mode_on_log_probabilities():
    c = wl.make_case(wl.config(2, vocab=500, prefix=(16, 16), n=(40, 40)), parts=("accept",))
    lg = dict(c)
    lg["kind"] = "logits"
    lg["target"] = np.log(c["target"].astype(np.float64)).astype(F32)
    a, b = oracle.accept(c), oracle.accept(lg)
    rel = np.abs(a["pq"][:, 0].astype(float) - b["pq"][:, 0]) / np.maximum(a["pq"][:, 0], 1e-30)
    assert rel.max() < 2e-6
    assert np.array_equal(a["accepted_len"], b["accepted_len"])
    assert np.array_equal(a["path"], b["path"])
    assert np.array_equal(a["bonus_token"], b["bonus_token"])


# ---------------------------------------------------------------- lossless
def test_lossless_first_token_distribution_and_alpha():
    """Chains of one draft token x ~ q: the emitted token (x if accepted, else
    the bonus) follows p (chi-square), and P(accept) = sum_x min(p, q)."""
    from scipy.stats import chisquare
    g = wl.rng(11, 11)
    V, n = 16, 200_000
    p = wl._softmax32(g.normal(0, 1, (1, V)))[0]
    q = wl._softmax32(g.normal(0, 1, (1, V)))[0]
    qn = q.astype(float) / q.astype(float).sum()
    x = g.choice(V, size=n, p=qn)
    T = np.tile(np.stack([p, p]), (n, 1))
    D = np.tile(np.stack([q, q]), (n, 1))
    toks = np.stack([np.full(n, -1), x], 1).ravel()
    U = (g.integers(0, 1 << 24, 2 * n) * 2.0 ** -24).astype(F32)
    case = accept_case([[-1, 0]] * n, V, T, D, toks, U)
    out = oracle.accept(case)
    emitted = np.where(out["accepted_len"] == 1, x, out["bonus_token"])
    counts = np.bincount(emitted, minlength=V)
    pn = p.astype(float) / p.astype(float).sum()
    assert chisquare(counts, pn * n).pvalue > 1e-3
    alpha = np.minimum(pn, qn).sum()
    acc = out["accepted_len"].mean()
    assert abs(acc - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / n)


# ---------------------------------------------------------------- golden
def test_golden_hand_worked_examples():
    for name in sorted(os.listdir(GOLDEN)):
        if not name.startswith("accept_") or not name.endswith(".json"):
            continue
        ex = json.load(open(os.path.join(GOLDEN, name)))
        case = accept_case([ex["parent"]], ex["vocab"], ex["target"], ex["draft"],
                           ex["tokens"], ex["uniforms"],
                           mask=None if ex.get("mask") is None else np.asarray(ex["mask"], np.uint32))
        checks = [(ex.get("test", 0), ex["expect"])]
        if "expect_ratio_test" in ex:
            checks.append((0, ex["expect_ratio_test"]))
        for test, want in checks:
            out = oracle.accept(case, test=test)
            assert out["accepted_len"][0] == want["accepted_len"], (name, test)
            assert list(out["path"][0, : want["accepted_len"]]) == want["path"], (name, test)
            assert out["bonus_token"][0] == want["bonus_token"], (name, test)
