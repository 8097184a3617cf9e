"""The synthetic workloads follow their stated recipe (CPU only): batch,
heads, head size, prefix lengths, tree sizes and depths, breadth-first
numbering with siblings in descending draft probability, the page table,
the multimodal prefix's image-token spread, the vocabulary sizes and the
uniforms' grid."""
import numpy as np
import pytest

from speculative_decoding_tree_attention_gb300 import workloads as wl


def depths(parent):
    d = np.zeros(len(parent), np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def trees(case):
    off = case["node_offsets"]
    return [case["parent"][off[b]:off[b + 1]] for b in range(case["batch"])]


RECIPE = {  # config: (batch, hq, hkv, d, prefix range, nodes range, max depth, vocab)
    1: (1, 4, 4, 64, (128, 128), (15, 15), 3, 1000),
    2: (1, 32, 32, 128, (1024, 1024), (64, 64), 6, 32000),
    3: (16, 32, 8, 128, (512, 4096), (26, 64), 5, 32000),
    4: (4, 28, 4, 128, (1600, 1600), (128, 128), 8, 151936),
    5: (4, 64, 8, 128, (32768, 32768), (256, 256), 10, 128256),
}


@pytest.mark.parametrize("num", [1, 2, 3, 4, 5])
def test_shapes_and_trees(num):
    B, hq, hkv, d, (plo, phi), (nlo, nhi), dmax, V = RECIPE[num]
    cfg = wl.config(num)
    assert (cfg["batch"], cfg["hq"], cfg["hkv"], cfg["d"], cfg["vocab"]) == (B, hq, hkv, d, V)
    case = wl.make_case(cfg, parts=())
    assert case["batch"] == B
    for par in trees(case):
        n = len(par)
        assert nlo <= n <= nhi
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, n))
        assert depths(par).max() <= dmax
        # breadth-first numbering: depth never decreases with the index
        assert np.all(np.diff(depths(par)) >= 0)
    if num == 1:  # the full binary tree of depth 3
        assert list(trees(case)[0]) == [-1] + [(i - 1) // 2 for i in range(1, 15)]


@pytest.mark.parametrize("num", [1, 3])
def test_prefix_lengths_and_page_table(num):
    B, _, hkv, d, (plo, phi), _, _, _ = RECIPE[num]
    case = wl.make_case(wl.config(num), parts=("attn",))
    lens = case["prefix_lens"]
    assert lens.shape == (B,) and lens.min() >= plo and lens.max() <= phi
    pages = np.concatenate([case["block_table"][b, : (lens[b] + 15) // 16] for b in range(B)])
    # every page of the pool is used exactly once (stored once, reached by index)
    assert np.array_equal(np.sort(pages), np.arange(case["num_blocks"]))
    if num == 3:  # shuffled: the table is not the identity order
        assert not np.array_equal(pages, np.arange(case["num_blocks"]))
    q = wl.bf16_bits_to_f32(case["q"]).astype(np.float64)
    assert q.shape == (int(case["node_offsets"][-1]), case["num_q_heads"], d)
    assert abs(q.std() - 1.0) < 0.05 and abs(q.mean()) < 0.05


def test_multimodal_image_tokens_have_the_larger_spread():
    case = wl.make_case(wl.config(4, batch=1), parts=("attn",))
    kp = wl.bf16_bits_to_f32(case["k_prefix"]).astype(np.float64)
    table = case["block_table"][0]
    rows = np.stack([kp[table[t // 16], :, t % 16] for t in range(1600)])  # [token][head][d]
    assert abs(rows[:576].std() - 2.0) < 0.05
    assert abs(rows[576:].std() - 1.0) < 0.03


@pytest.mark.parametrize("num", [2, 3])
def test_children_in_descending_draft_probability(num):
    case = wl.make_case(wl.config(num, batch=2) if num == 3 else wl.config(num),
                        parts=("accept",), kind="probs")
    off = case["node_offsets"]
    for b in range(case["batch"]):
        par = case["parent"][off[b]:off[b + 1]]
        tok = case["draft_tokens"][off[b]:off[b + 1]]
        for j in range(len(par)):
            kids = [i for i in range(j + 1, len(par)) if par[i] == j]
            q = case["draft_probs"][off[b] + j]
            pk = [q[tok[i]] for i in kids]
            assert pk == sorted(pk, reverse=True)
            assert len(set(tok[i] for i in kids)) == len(kids)  # distinct tokens
    u = case["uniforms"].astype(np.float64) * 2.0 ** 24
    assert np.all(u == np.floor(u)) and np.all(u < 2.0 ** 24)
