"""Pins of the oracle's commit of the accepted path (CPU only).

The commit is a copy, so it is pinned by what the copy must achieve rather
than by retyping it:
  * re-reading the pool through the block table at positions L .. L+a gives
    the root's and the accepted nodes' K/V rows in path order, and no other
    pool row changes;
  * attention agrees across the commit: an accepted node at depth d attends,
    in the verification step, to the prefix, its ancestors and itself; after
    the commit the same query as a one-node tree over the first L+d
    committed positions sees exactly the same keys, so the fp64 attention
    oracle gives the same output;
  * malformed paths, failed accept passes and missing pages leave everything
    unchanged, with the documented status."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl


def _case(num=1, **over):
    return wl.make_case(wl.config(num, **over), parts=("attn",))


def _first_child_path(parent, n0, N, depth):
    """Root-down path following the first child at each level."""
    path, cur = [], 0
    for _ in range(depth):
        kids = [v for v in range(1, N) if parent[n0 + v] == cur]
        if not kids:
            break
        cur = kids[0]
        path.append(cur)
    return path


def _setup(case, depths):
    B, maxn = case["batch"], case["max_nodes"]
    off = case["node_offsets"]
    kp, vp, table = wl.extend_pool(case, maxn + 1)
    path = np.full((B, maxn), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        p = _first_child_path(case["parent"], off[b], off[b + 1] - off[b], depths[b])
        path[b, : len(p)] = p
        acc[b] = len(p)
    return kp, vp, table, path, acc


def _commit(case, kp, vp, table, path, acc, lens=None):
    return oracle.commit_kv(case["k_nodes"], case["v_nodes"], case["parent"],
                            case["node_offsets"], acc, path, table,
                            case["prefix_lens"] if lens is None else lens, kp, vp,
                            case["max_nodes"])


@pytest.mark.parametrize("num, over, depths", [
    (1, {}, [3]),                                             # binary tree, full depth
    (1, {}, [0]),                                             # root only
    (3, dict(batch=3, hq=4, hkv=2, d=64, prefix=(17, 70), n=(5, 12)), [2, 0, 4]),
])
def test_commit_rereads_through_block_table(num, over, depths):
    case = _case(num, **over)
    kp, vp, table, path, acc = _setup(case, depths)
    k2, v2, new, st = _commit(case, kp, vp, table, path, acc)
    assert np.all(st == 0)
    assert np.array_equal(new, case["prefix_lens"] + acc + 1)
    touched = np.zeros(kp.shape[:1] + kp.shape[2:3], bool)  # [page][row]
    off = case["node_offsets"]
    for b in range(case["batch"]):
        L = int(case["prefix_lens"][b])
        nodes = [0] + list(path[b, : acc[b]])
        for t, v in enumerate(nodes):
            pg, row = table[b, (L + t) // 16], (L + t) % 16
            assert np.array_equal(k2[pg, :, row], case["k_nodes"][off[b] + v])
            assert np.array_equal(v2[pg, :, row], case["v_nodes"][off[b] + v])
            touched[pg, row] = True
    untouched = ~touched
    assert np.array_equal(k2.transpose(0, 2, 1, 3)[untouched], kp.transpose(0, 2, 1, 3)[untouched])
    assert np.array_equal(v2.transpose(0, 2, 1, 3)[untouched], vp.transpose(0, 2, 1, 3)[untouched])


def test_attention_agrees_across_the_commit():
    case = _case(3, batch=2, hq=4, hkv=2, d=64, prefix=(30, 50), n=(7, 12), depth=4)
    kp, vp, table, path, acc = _setup(case, [4, 4])
    k2, v2, new, st = _commit(case, kp, vp, table, path, acc)
    assert np.all(st == 0)
    off = case["node_offsets"]
    for b in range(case["batch"]):
        L = int(case["prefix_lens"][b])
        for d in range(1, int(acc[b]) + 1):
            v = int(path[b, d - 1])
            rows = np.array([(b, v, h) for h in range(case["num_q_heads"])], np.int32)
            before = oracle.tree_attention_rows(case, rows)
            # one-node tree: query and key of node v, prefix = first L + d
            # committed positions (old prefix, root, path[0 .. d-2])
            one = dict(batch=1, num_q_heads=case["num_q_heads"], num_kv_heads=case["num_kv_heads"],
                       head_dim=case["head_dim"], block_size=16, softmax_scale=case["softmax_scale"],
                       q=case["q"][off[b] + v][None], k_nodes=case["k_nodes"][off[b] + v][None],
                       v_nodes=case["v_nodes"][off[b] + v][None], parent=np.array([-1], np.int32),
                       node_offsets=np.array([0, 1], np.int32),
                       prefix_lens=np.array([L + d], np.int32), block_table=table[b][None],
                       k_prefix=k2, v_prefix=v2)
            after = oracle.tree_attention_rows(
                one, np.array([(0, 0, h) for h in range(case["num_q_heads"])], np.int32))
            np.testing.assert_allclose(after, before, rtol=1e-12, atol=1e-12)


def test_failures_leave_everything_unchanged():
    case = _case(3, batch=4, hq=4, hkv=2, d=64, prefix=(40, 60), n=(6, 10))
    kp, vp, table, path, acc = _setup(case, [2, 2, 2, 2])
    acc, path, table = acc.copy(), path.copy(), table.copy()
    lens = np.array(case["prefix_lens"], np.int32, copy=True)
    acc[0] = -1                                                  # accept pass failed
    path[1, 1] = path[1, 0]                                      # not a child of path[1, 0]
    acc[2] = case["node_offsets"][3] - case["node_offsets"][2]   # a >= N
    lens[3] = 31                                                 # positions 31 .. 33
    table[3, 2] = -1                                             # no page for 32, 33
    k2, v2, new, st = _commit(case, kp, vp, table, path, acc, lens)
    assert list(st) == [5, 5, 5, 7]
    assert np.array_equal(new, lens)
    assert np.array_equal(k2, kp) and np.array_equal(v2, vp)
    # the same sequence 3 with its page restored commits
    table[3, 2] = kp.shape[0] - 1
    k3, v3, new3, st3 = _commit(case, kp, vp, table, path, acc, lens)
    assert list(st3) == [5, 5, 5, 0] and new3[3] == 31 + acc[3] + 1
