"""GPU parity of tv_commit_kv against the oracle's commit: the written pool
pages, the new prefix lengths and the status must match bit for bit (a copy
has nothing to round).  Paths come from a root-down walk of each tree, or
from the accept pass itself (GPU accept feeding GPU commit, against oracle
accept feeding oracle commit)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import ensure_built, run_accept

pytestmark = pytest.mark.gpu


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _i32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def _paths(case, depth_of, seed):
    g = np.random.default_rng(seed)
    B, maxn = case["batch"], case["max_nodes"]
    off, par = case["node_offsets"], case["parent"]
    path = np.full((B, maxn), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        cur, p = 0, []
        for _ in range(depth_of(b)):
            kids = [v for v in range(1, off[b + 1] - off[b]) if par[off[b] + v] == cur]
            if not kids:
                break
            cur = int(g.choice(kids))
            p.append(cur)
        path[b, : len(p)] = p
        acc[b] = len(p)
    return path, acc


def _run_both(case, kp, vp, table, path, acc, lens=None):
    lens = case["prefix_lens"] if lens is None else lens
    ref = oracle.commit_kv(case["k_nodes"], case["v_nodes"], case["parent"], case["node_offsets"],
                           acc, path, table, lens, kp, vp, case["max_nodes"])
    k_pool, v_pool = _bf16(kp), _bf16(vp)
    new, st = tv.commit_kv(_bf16(case["k_nodes"]), _bf16(case["v_nodes"]), _i32(case["parent"]),
                           _i32(case["node_offsets"]), _i32(acc), _i32(path), _i32(table),
                           _i32(lens), k_pool, v_pool, max_nodes=int(case["max_nodes"]))
    torch.cuda.synchronize()
    got = (k_pool.view(torch.int16).cpu().numpy().view(np.uint16),
           v_pool.view(torch.int16).cpu().numpy().view(np.uint16),
           new.cpu().numpy(), st.cpu().numpy())
    return got, ref


def _assert_same(got, ref):
    assert np.array_equal(got[3], ref[3]), (got[3], ref[3])
    assert np.array_equal(got[2], ref[2])
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("num, over", [
    (3, dict(batch=6, prefix=(300, 3000), n=(5, 64))),            # shuffled pages, D=128, GQA
    (1, dict()),                                                   # D=64, binary tree
    (3, dict(batch=5, hq=8, hkv=8, d=64, prefix=(1, 40), n=(1, 9))),  # tiny prefixes, 1-node trees
])
def test_commit_bit_exact(num, over):
    ensure_built()
    case = wl.make_case(wl.config(num, **over), parts=("attn",))
    kp, vp, table = wl.extend_pool(case, case["max_nodes"] + 1)
    path, acc = _paths(case, lambda b: 2 + 3 * b, seed=num)
    got, ref = _run_both(case, kp, vp, table, path, acc)
    assert np.all(ref[3] == 0)
    _assert_same(got, ref)


def test_commit_statuses():
    ensure_built()
    case = wl.make_case(wl.config(3, batch=5, hq=8, hkv=2, d=128, prefix=(40, 60), n=(6, 10)),
                        parts=("attn",))
    kp, vp, table = wl.extend_pool(case, case["max_nodes"] + 1)
    path, acc = _paths(case, lambda b: 2, seed=7)
    lens = np.array(case["prefix_lens"], np.int32, copy=True)
    acc[0] = -1                                                   # failed accept pass
    path[1, 1] = path[1, 0]                                       # not a child
    acc[2] = case["node_offsets"][3] - case["node_offsets"][2]    # a >= N
    lens[3] = 31
    table[3, 2] = -1                                              # no page for 32, 33
    got, ref = _run_both(case, kp, vp, table, path, acc, lens)
    assert list(ref[3]) == [5, 5, 5, 7, 0]
    _assert_same(got, ref)


def test_accept_then_commit_on_device():
    ensure_built()
    case = wl.make_case(wl.config(3, batch=4, prefix=(100, 900), n=(20, 40), vocab=3000),
                        parts=("attn", "accept"), kind="probs")
    kp, vp, table = wl.extend_pool(case, case["max_nodes"] + 1)
    gacc = run_accept(case)
    racc = oracle.accept(case)
    assert np.array_equal(gacc["accepted_len"], racc["accepted_len"])
    path = np.ascontiguousarray(gacc["path"], np.int32)
    got, ref = _run_both(case, kp, vp, table, path, gacc["accepted_len"])
    assert np.all(ref[3] == 0)
    _assert_same(got, ref)
    assert np.array_equal(got[2], case["prefix_lens"] + racc["accepted_len"] + 1)
