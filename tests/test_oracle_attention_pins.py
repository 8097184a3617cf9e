"""Pins of the fp64 attention oracle against facts the pages and mathematics fix.

The tree mask of the edge-cloud tree-attention page (§2.2.2): node i sees tree
node j iff j is an ancestor of i or j == i; the committed prefix is stored once
and reached through the block table (multimodal pruning page §3.2, common-prefix
merging).  Each pin below checks the oracle with an independent route:
closed forms, a library attention routine (torch SDPA, fp64, CPU) on gathered
keys, brute force over every small tree, and invariances.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl

BS = 16


def bits(x):
    return wl.to_bf16_bits(np.asarray(x, dtype=np.float32))


def f64(b):
    return wl.bf16_bits_to_f32(b).astype(np.float64)


def attn_case(parents, prefix_lens, hq=4, hkv=2, d=64, seed=1, shuffle=False, scale=0.0):
    """Random bf16 case for explicit trees (one parent list per sequence)."""
    B = len(parents)
    ns = [len(p) for p in parents]
    off = np.zeros(B + 1, np.int32)
    off[1:] = np.cumsum(ns)
    tot = int(off[-1])
    nblk = [(l + BS - 1) // BS for l in prefix_lens]
    nb = max(1, sum(nblk))
    perm = np.arange(nb, dtype=np.int32)
    if shuffle:
        perm = wl.rng(seed, 99).permutation(nb).astype(np.int32)
    table = np.zeros((B, max(1, max(nblk))), np.int32)
    pos = 0
    for b in range(B):
        table[b, : nblk[b]] = perm[pos: pos + nblk[b]]
        pos += nblk[b]
    g = wl.rng(seed, 7)
    return dict(batch=B, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=BS,
                block_table=table, prefix_lens=np.asarray(prefix_lens, np.int32),
                node_offsets=off, parent=np.concatenate([np.asarray(p, np.int32) for p in parents]),
                q=bits(g.standard_normal((tot, hq, d))),
                k_prefix=bits(g.standard_normal((nb, hkv, BS, d))),
                v_prefix=bits(g.standard_normal((nb, hkv, BS, d))),
                k_nodes=bits(g.standard_normal((tot, hkv, d))),
                v_nodes=bits(g.standard_normal((tot, hkv, d))), softmax_scale=scale)


def prefix_kv(case, b, kvh, which):
    """Logical prefix keys/values of sequence b, gathered through the table."""
    L = int(case["prefix_lens"][b])
    pool = case["k_prefix" if which == "k" else "v_prefix"]
    out = np.zeros((L, case["head_dim"]))
    for t in range(L):
        out[t] = f64(pool[case["block_table"][b, t // BS], kvh, t % BS])
    return out


def ancestors_closure(par):
    """Ancestor-or-self relation by Warshall transitive closure of the parent edge."""
    n = len(par)
    R = np.eye(n, dtype=bool)
    for i in range(1, n):
        R[i, par[i]] = True
    for k in range(n):
        R |= R[:, k:k + 1] & R[k:k + 1, :]
    return R  # R[i, j]: j is an ancestor of i or j == i


def all_trees(n):
    for choice in itertools.product(*[range(i) for i in range(1, n)]):
        yield [-1] + list(choice)


def random_tree(n, g):
    return [-1] + [int(g.integers(0, i)) for i in range(1, n)]


# ----------------------------------------------------------------------------
def test_mask_closed_form_all_small_trees():
    """Q = 0 makes every visible key equally weighted: with prefix V = e_{D-1}
    and node V_j = e_j, output i is exactly [j visible]/(L + #visible nodes) in
    column j and L/(L + #visible) in the last column.  All 154 trees with up to
    6 nodes, ancestry by transitive closure."""
    trees = [t for n in range(1, 7) for t in all_trees(n)]
    assert len(trees) == 1 + 1 + 2 + 6 + 24 + 120
    L = 21
    case = attn_case(trees, [L] * len(trees), hq=2, hkv=1, d=16)
    case["q"][:] = 0
    case["v_prefix"][:] = 0
    case["v_prefix"][..., 15] = bits(1.0)
    case["v_nodes"][:] = 0
    off = case["node_offsets"]
    for b, par in enumerate(trees):
        for j in range(len(par)):
            case["v_nodes"][off[b] + j, :, j] = bits(1.0)
    out = oracle.tree_attention(case)
    for b, par in enumerate(trees):
        R = ancestors_closure(par)
        for i in range(len(par)):
            cnt = L + R[i].sum()
            exp_row = np.zeros(16)
            exp_row[: len(par)] = R[i] / cnt
            exp_row[15] = L / cnt
            for h in range(2):
                np.testing.assert_allclose(out[off[b] + i, h], exp_row, rtol=0, atol=1e-15)


def _sdpa(q, k, v, scale, mask=None):
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    m = None if mask is None else torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m,
                                                            scale=scale)[0, 0].numpy()


def test_chain_tree_is_causal_attention_sdpa():
    """A chain (parent(i) = i-1) is ordinary causal attention over [prefix; nodes]
    (the single-chain special case of tree verification)."""
    N, L = 12, 37
    case = attn_case([[-1] + list(range(N - 1))], [L], hq=4, hkv=2, d=64, seed=3)
    out = oracle.tree_attention(case)
    scale = 1 / math.sqrt(64)
    mask = np.ones((N, L + N), dtype=bool)
    mask[:, L:] = np.tril(np.ones((N, N), dtype=bool))
    for h in range(4):
        kvh = h // 2
        k = np.concatenate([prefix_kv(case, 0, kvh, "k"), f64(case["k_nodes"][:, kvh])])
        v = np.concatenate([prefix_kv(case, 0, kvh, "v"), f64(case["v_nodes"][:, kvh])])
        ref = _sdpa(f64(case["q"][:, h]), k, v, scale, mask)
        np.testing.assert_allclose(out[:, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_node_output_is_attention_over_its_root_path(seed):
    """Each node's output equals plain (unmasked) attention of its query over the
    prefix followed by the keys of its own root-to-node path, gathered by
    walking up the parents."""
    g = wl.rng(seed, 5)
    parents = [random_tree(int(g.integers(1, 30)), g) for _ in range(3)]
    lens = [int(g.integers(0, 70)) for _ in range(3)]
    case = attn_case(parents, lens, hq=6, hkv=3, d=32, seed=seed)
    out = oracle.tree_attention(case)
    off = case["node_offsets"]
    scale = 1 / math.sqrt(32)
    for b, par in enumerate(parents):
        for i in range(len(par)):
            path = []
            k_ = i
            while k_ >= 0:
                path.append(k_)
                k_ = par[k_]
            path = path[::-1]
            for h in range(6):
                kvh = h // 2
                k = np.concatenate([prefix_kv(case, b, kvh, "k"),
                                    f64(case["k_nodes"][off[b] + np.array(path), kvh])])
                v = np.concatenate([prefix_kv(case, b, kvh, "v"),
                                    f64(case["v_nodes"][off[b] + np.array(path), kvh])])
                ref = _sdpa(f64(case["q"][off[b] + i, h])[None], k, v, scale)[0]
                np.testing.assert_allclose(out[off[b] + i, h], ref, rtol=0, atol=1e-12)


def test_block_table_shuffle_is_bit_identical():
    """The same logical prefix stored in permuted pages gives identical outputs."""
    parents = [random_tree(9, wl.rng(1, 1)), random_tree(4, wl.rng(1, 2))]
    a = attn_case(parents, [50, 33], seed=11)
    b = dict(a)
    nb = a["k_prefix"].shape[0]
    perm = wl.rng(4, 4).permutation(nb)
    kp = np.empty_like(a["k_prefix"])
    vp = np.empty_like(a["v_prefix"])
    kp[perm] = a["k_prefix"]
    vp[perm] = a["v_prefix"]
    b["k_prefix"], b["v_prefix"] = kp, vp
    b["block_table"] = perm[a["block_table"]].astype(np.int32)
    assert np.array_equal(oracle.tree_attention(a), oracle.tree_attention(b))


def test_topological_relabelling_permutes_outputs():
    par = [-1, 0, 0, 1, 1, 2, 3, 3, 5]
    # new label of old node i; keeps parents before children
    new_of = [0, 2, 1, 4, 3, 5, 7, 8, 6]
    new_par = [0] * 9
    for i, p in enumerate(par):
        new_par[new_of[i]] = -1 if p < 0 else new_of[p]
    assert all(new_par[i] < i for i in range(1, 9))
    a = attn_case([par], [40], seed=21)
    b = dict(a)
    inv = np.argsort(new_of)
    b["parent"] = np.asarray(new_par, np.int32)
    for key in ("q", "k_nodes", "v_nodes"):
        b[key] = a[key][inv]
    oa, ob = oracle.tree_attention(a), oracle.tree_attention(b)
    np.testing.assert_allclose(ob[new_of], oa, rtol=0, atol=1e-13)


def test_gqa_grouping_is_contiguous():
    """Query head h reads KV head floor(h / (Hq/Hkv)): with Q = 0 and every value
    of KV head c equal to c+1, output head h is exactly floor(h/g)+1."""
    case = attn_case([[-1, 0, 1, 1]], [19], hq=8, hkv=4, d=16)
    case["q"][:] = 0
    for c in range(4):
        case["v_prefix"][:, c] = bits(c + 1.0)
        case["v_nodes"][:, c] = bits(c + 1.0)
    out = oracle.tree_attention(case)
    for h in range(8):
        np.testing.assert_allclose(out[:, h], h // 2 + 1, rtol=1e-15, atol=0)


@pytest.mark.parametrize("scale", [0.0, 0.37])
def test_two_key_closed_form(scale):
    """Prefix of one key and a root-only tree: a two-way softmax by hand."""
    case = attn_case([[-1]], [1], hq=1, hkv=1, d=8, seed=5, scale=scale)
    out = oracle.tree_attention(case)[0, 0]
    sc = scale if scale else 1 / math.sqrt(8)
    q = f64(case["q"][0, 0])
    k0, v0 = f64(case["k_prefix"][0, 0, 0]), f64(case["v_prefix"][0, 0, 0])
    k1, v1 = f64(case["k_nodes"][0, 0]), f64(case["v_nodes"][0, 0])
    s0, s1 = sc * float(q @ k0), sc * float(q @ k1)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    np.testing.assert_allclose(out, w0 * v0 + (1 - w0) * v1, rtol=0, atol=1e-14)


def test_empty_prefix_root_only_returns_root_value():
    case = attn_case([[-1], [-1, 0]], [0, 0], hq=2, hkv=1, d=16, seed=8)
    out = oracle.tree_attention(case)
    assert np.array_equal(out[0, 0], f64(case["v_nodes"][0, 0]))
    assert np.array_equal(out[1, 1], f64(case["v_nodes"][1, 0]))


def test_single_node_is_decode_attention():
    """N = 1 (the root only) is ordinary decode attention over prefix + itself."""
    case = attn_case([[-1]], [45], hq=2, hkv=2, d=32, seed=9)
    out = oracle.tree_attention(case)
    for h in range(2):
        k = np.concatenate([prefix_kv(case, 0, h, "k"), f64(case["k_nodes"][:, h])])
        v = np.concatenate([prefix_kv(case, 0, h, "v"), f64(case["v_nodes"][:, h])])
        ref = _sdpa(f64(case["q"][0, h])[None], k, v, 1 / math.sqrt(32))[0]
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-12)


def test_sampled_rows_match_full():
    parents = [random_tree(11, wl.rng(2, 2))]
    case = attn_case(parents, [30], seed=4)
    full = oracle.tree_attention(case)
    rows = np.array([[0, 3, 1], [0, 10, 3], [0, 0, 0]], np.int32)
    part = oracle.tree_attention_rows(case, rows)
    for r, (b, i, h) in enumerate(rows):
        assert np.array_equal(part[r], full[i, h])
