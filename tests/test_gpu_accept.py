"""GPU parity of tv_accept (through the C ABI) against the oracle.

Probability inputs (with or without the pruning mask): bit-exact accepted
length, path, bonus token, status and the (p~, q~) of every test.
Logits inputs: the GPU's fp32 softmax and the oracle's fp64 one differ by
rounding, so p~ agrees to 1e-5 relative and q~ bit for bit.  A tree's
outputs may differ from the oracle's only where a declared near-tie explains
it: a tested node whose decision differs must have |u q~ - p~| within the p~
tolerance, and with every decision equal the path must be equal and a
different bonus token needs t = floor(u_0 S) within the tolerance of a
boundary of the cut node's cumulative sums.  Every such tree is counted.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import run_accept

pytestmark = pytest.mark.gpu

PQ_RTOL = 1e-5


def assert_bit_exact(case, gpu, ref, what):
    assert np.array_equal(gpu["status"], ref["status"]), what
    assert np.array_equal(gpu["accepted_len"], ref["accepted_len"]), what
    assert np.array_equal(gpu["path"], ref["path"]), what
    assert np.array_equal(gpu["bonus_token"], ref["bonus_token"]), what
    tot = int(case["node_offsets"][-1])
    assert np.array_equal(gpu["debug_pq"][:tot].view(np.uint32), ref["pq"][:tot].view(np.uint32)), what


@pytest.mark.parametrize("num", [1, 2, 3, 4, 5])
def test_full_size_probs_bit_exact(num):
    case = wl.make_case(wl.config(num), parts=("accept",), kind="probs")
    gpu = run_accept(case)
    ref = oracle.accept(case)
    assert_bit_exact(case, gpu, ref, f"config {num} probs")


def test_multimodal_without_mask_bit_exact():
    case = wl.make_case(wl.config(4), parts=("accept",), kind="probs")
    case["retained_mask"] = None
    assert_bit_exact(case, run_accept(case), oracle.accept(case), "config 4 no mask")


def near_tie_nodes(case, pq):
    u = case["uniforms"]
    gap = np.abs(u.astype(np.float64) * pq[:, 1] - pq[:, 0])
    return gap <= 4 * PQ_RTOL * np.maximum(np.abs(pq[:, 0]), 1e-30)


def decisions(case, pq):
    """The ratio test fl32(u q~) < p~ of every node from a (p~, q~) table."""
    u = case["uniforms"].astype(np.float32)
    return (u * pq[:, 1].astype(np.float32)) < pq[:, 0].astype(np.float32)


def bonus_near_tie(case, b, cut, eps):
    """True when the bonus draw of tree b at local cut node `cut` lies near a
    boundary of the quantised cumulative sums: a relative change of at most
    `eps` in every target probability moves a partial sum C and
    t = floor(u_0 S) by at most eps*C and eps*t, so the token can only move
    when |t - C| <= 4 eps (t + C) at the drawn token's lower or upper
    boundary (factor 4: margin)."""
    off = case["node_offsets"]
    n0, n1 = int(off[b]), int(off[b + 1])
    par = case["parent"][n0:n1]
    row = n0 + cut
    V = case["vocab"]
    x = case["target"][row].astype(np.float64)
    p = np.exp(x - x.max())
    p = (p / p.sum()).astype(np.float32)
    q = case["draft_probs"][row].astype(np.float32)
    m = case.get("retained_mask")
    if m is not None:
        bits = ((m[row][np.arange(V) // 32] >> (np.arange(V) % 32).astype(np.uint32)) & 1).astype(bool)
        qq = np.clip(np.where(bits & (q > 0), q, 0.0), 0, 32).astype(np.float64)
        z = np.float32(np.floor(qq * 2.0 ** 40).sum()) * np.float32(2.0 ** -40)
        p = np.where(bits, p / z, 0).astype(np.float32)
        q = np.where(bits, q / z, 0).astype(np.float32)
    two40 = 2.0 ** 40
    has_children = bool(np.any(par[cut + 1:] == cut))
    for r in ([(p - q).astype(np.float32)] if has_children else []) + [p]:
        f = np.floor(np.clip(np.nan_to_num(r.astype(np.float64)), 0, 32) * two40)
        S = f.sum()
        if S <= 0:
            continue
        t = np.floor(float(case["uniforms"][n0]) * S)
        cum = np.cumsum(f)
        k = int(np.searchsorted(cum, t, side="right"))
        lo = cum[k - 1] if k > 0 else 0.0
        hi = cum[min(k, V - 1)]
        return bool(t - lo <= 4 * eps * (t + lo) or hi - t <= 4 * eps * (t + hi))
    return True  # argmax fallback: no draw to compare


@pytest.mark.parametrize("num", [1, 2, 3, 4, 5])
def test_full_size_logits_within_tolerance(num):
    case = wl.make_case(wl.config(num), parts=("accept",), kind="logits")
    gpu = run_accept(case)
    ref = oracle.accept(case)
    assert np.all(gpu["status"] == 0)
    tot = int(case["node_offsets"][-1])
    gp, rp = gpu["debug_pq"][:tot].astype(np.float64), ref["pq"][:tot].astype(np.float64)
    rel = np.abs(gp - rp) / np.maximum(np.abs(rp), 1e-30)
    assert rel[:, 0].max() <= PQ_RTOL and np.array_equal(gp[:, 1], rp[:, 1])
    eps = max(float(rel[:, 0].max()), 1e-7)  # measured p~ error (floor: a few fp32 ulps)
    ties = near_tie_nodes(case, rp)
    dg, dr = decisions(case, gp), decisions(case, rp)
    off = case["node_offsets"]
    explained = 0
    for b in range(case["batch"]):
        same = (gpu["accepted_len"][b] == ref["accepted_len"][b] and
                np.array_equal(gpu["path"][b], ref["path"][b]) and
                gpu["bonus_token"][b] == ref["bonus_token"][b])
        sl = slice(off[b] + 1, off[b + 1])
        flips = np.nonzero(dg[sl] != dr[sl])[0]
        assert np.all(ties[sl][flips]), f"tree {b}: a decision differs without a near-tie"
        if same:
            continue
        explained += 1
        if flips.size:
            continue  # a near-tie decision moved the walk: anything downstream may differ
        assert gpu["accepted_len"][b] == ref["accepted_len"][b] and \
            np.array_equal(gpu["path"][b], ref["path"][b]), \
            f"tree {b}: equal decisions but a different path"
        cut = int(ref["path"][b][ref["accepted_len"][b] - 1]) if ref["accepted_len"][b] > 0 else 0
        assert bonus_near_tie(case, b, cut, eps), f"tree {b}: bonus differs without a near-tie"
    print(f"config {num} logits: {explained} tree(s) differ, each at a declared near-tie")


# ---------------------------------------------------------------- edge cases
def random_forest(seed, n_trees, V, nmax, chain=False, mask_frac=None):
    g = wl.rng(seed, 77)
    parents, T, D, toks, U = [], [], [], [], []
    for _ in range(n_trees):
        n = int(g.integers(1, nmax + 1))
        par = [-1] + ([i - 1 for i in range(1, n)] if chain else
                      [int(g.integers(0, i)) for i in range(1, n)])
        P = wl._softmax32(g.normal(0, 1.2, (n, V)))
        Q = wl._softmax32(P.astype(np.float64) * 0 + g.normal(0, 1.2, (n, V)))
        tk = [-1] + [int(np.argmax(Q[par[i]] + g.random(V) * 0.05)) for i in range(1, n)]
        parents.append(par), T.append(P), D.append(Q), toks.extend(tk)
        U.extend((g.integers(0, 1 << 24, n) * 2.0 ** -24).astype(np.float32))
    off = np.zeros(n_trees + 1, np.int32)
    off[1:] = np.cumsum([len(p) for p in parents])
    case = dict(node_offsets=off, parent=np.concatenate([np.asarray(p, np.int32) for p in parents]),
                vocab=V, target=np.concatenate(T), draft_probs=np.concatenate(D),
                draft_tokens=np.asarray(toks, np.int32), uniforms=np.asarray(U, np.float32),
                retained_mask=None, kind="probs", max_nodes=nmax, batch=n_trees)
    if mask_frac is not None:
        W = (V + 31) // 32
        bits = g.random((off[-1], W * 32)) < mask_frac
        words = np.zeros((off[-1], W), np.uint64)
        for k in range(32):
            words |= bits[:, k::32].astype(np.uint64) << np.uint64(k)
        case["retained_mask"] = words.astype(np.uint32)
    return case


@pytest.mark.parametrize("V", [1, 3, 37, 1001, 16385, 40003])
@pytest.mark.parametrize("chain", [False, True])
def test_odd_vocab_sizes_and_alignment(V, chain):
    case = random_forest(V, 24, V, 9, chain=chain)
    assert_bit_exact(case, run_accept(case), oracle.accept(case), f"V={V}")


@pytest.mark.parametrize("V", [50, 20000])
def test_renorm_random_masks(V):
    case = random_forest(3 + V, 20, V, 12, mask_frac=0.4)
    assert_bit_exact(case, run_accept(case), oracle.accept(case), f"mask V={V}")


def test_large_trees_512_nodes():
    case = random_forest(9, 3, 300, 512)
    assert_bit_exact(case, run_accept(case), oracle.accept(case), "512 nodes")


def test_everything_accepted_and_nothing_accepted():
    V = 64
    case = random_forest(4, 6, V, 8, chain=True)
    case["uniforms"][:] = 0.0  # u = 0: accept wherever p > 0
    assert_bit_exact(case, run_accept(case), oracle.accept(case), "u=0")
    case["uniforms"][:] = np.float32(1 - 2 ** -24)
    assert_bit_exact(case, run_accept(case), oracle.accept(case), "u->1")


def test_bad_trees_report_status():
    case = random_forest(5, 4, 100, 6)
    off = case["node_offsets"]
    if off[2] - off[1] >= 2:
        case["parent"][off[1] + 1] = 5
    case["draft_tokens"][off[3] - 1] = 100 if off[3] - off[2] >= 2 else case["draft_tokens"][off[3] - 1]
    gpu, ref = run_accept(case), oracle.accept(case)
    assert np.array_equal(gpu["status"], ref["status"])
    assert np.array_equal(gpu["accepted_len"], ref["accepted_len"])
    assert np.array_equal(gpu["bonus_token"], ref["bonus_token"])
    assert np.array_equal(gpu["path"], ref["path"])


def test_zero_mass_rows_fall_back_to_argmax():
    V = 40
    case = random_forest(6, 3, V, 4)
    case["target"][:] = 0.0
    case["target"][:, 7] = 1e-13   # below the 2^-40 quantum
    case["target"][:, 9] = 1e-13
    assert_bit_exact(case, run_accept(case), oracle.accept(case), "argmax fallback")


def test_repeatable():
    case = wl.make_case(wl.config(2), parts=("accept",), kind="logits")
    a, b = run_accept(case), run_accept(case)
    for k in ("accepted_len", "path", "bonus_token", "debug_pq"):
        assert np.array_equal(a[k], b[k])
