"""GPU parity of the multi-candidate accept walk (test "multi") against the
oracle, through the C ABI.

Probability inputs (with or without the retained-set mask, with calibration
factors): bit-exact accepted length, path, bonus token, status and the
(cur(x), q~(x)) each tested child saw.  Logits inputs: the GPU's fp32 softmax
and the oracle's fp64 one differ by rounding, so decisions must agree on
every tree with no tested node near its acceptance boundary."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from test_gpu_accept import PQ_RTOL, assert_bit_exact, random_forest
from tv_testlib import accept_device, ensure_built

pytestmark = pytest.mark.gpu


def run_multi(case, gamma=None, test="multi"):
    ensure_built()
    t = accept_device(case)
    g = None if gamma is None else torch.from_numpy(np.ascontiguousarray(gamma, np.float32)).cuda()
    r = tv.accept(t["target"], t["draft"], t["tokens"], t["parent"], t["off"], t["uniforms"],
                  t["mask"], max_nodes=int(case["max_nodes"]), kind=case.get("kind", "probs"),
                  debug_pq=True, test=test, gamma=g)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in r.items()}


@pytest.mark.parametrize("num", [1, 2, 3, 4])
def test_full_size_probs_bit_exact(num):
    case = wl.make_case(wl.config(num), parts=("accept",), kind="probs")
    assert_bit_exact(case, run_multi(case), oracle.accept(case, test=2), f"config {num}")


def test_long_context_shape_bit_exact():
    case = wl.make_case(wl.config(5, batch=2), parts=("accept",), kind="probs")
    assert_bit_exact(case, run_multi(case), oracle.accept(case, test=2), "config 5, 2 trees")


@pytest.mark.parametrize("V", [1, 3, 37, 1001, 16385, 40003])
def test_odd_vocab_sizes_forests_and_chains(V):
    for chain in (False, True):
        case = random_forest(V + 7, 24, V, 9, chain=chain)
        assert_bit_exact(case, run_multi(case), oracle.accept(case, test=2), f"V={V} chain={chain}")


def test_chains_decide_as_the_ratio_test():
    case = random_forest(31, 24, 5000, 10, chain=True)
    a, b = run_multi(case, test="ratio"), run_multi(case)
    for k in ("accepted_len", "path", "bonus_token", "status"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("V", [50, 20000])
def test_retained_masks_and_gamma(V):
    case = random_forest(3 + V, 20, V, 12, mask_frac=0.4)
    gamma = np.random.default_rng(V).uniform(0.3, 3.0, case["batch"]).astype(np.float32)
    assert_bit_exact(case, run_multi(case, gamma=gamma), oracle.accept(case, test=2, gamma=gamma),
                     f"mask V={V}")


def test_many_rejections_and_wide_nodes():
    # wide roots with every child rejected (u -> 1), so the residual chain
    # runs through all siblings, and everything accepted (u = 0)
    V = 3000
    g = wl.rng(8, 601)
    parents = []
    for t in range(6):
        k = 24 + 4 * t
        parents.append([-1] + [0] * k + [1 + i for i in range(5)])
    n = [len(p) for p in parents]
    tot = sum(n)
    P = wl._softmax32(g.normal(0, 2.0, (tot, V)))
    Q = wl._softmax32(g.normal(0, 2.0, (tot, V)))
    toks = []
    for p in parents:
        toks += [-1] + [int(x) for x in g.integers(0, V, len(p) - 1)]
    from test_oracle_accept_pins import accept_case
    for u in (np.float32(1 - 2 ** -24), np.float32(0.0), None):
        U = (g.integers(0, 1 << 24, tot) * 2.0 ** -24).astype(np.float32) if u is None else \
            np.full(tot, u, np.float32)
        case = accept_case(parents, V, P, Q, toks, U)
        assert_bit_exact(case, run_multi(case), oracle.accept(case, test=2), f"u={u}")


def test_large_trees_512_nodes():
    case = random_forest(9, 3, 300, 512)
    assert_bit_exact(case, run_multi(case), oracle.accept(case, test=2), "512 nodes")


def test_bad_trees_report_status():
    case = random_forest(5, 4, 100, 6)
    off = case["node_offsets"]
    if off[2] - off[1] >= 2:
        case["parent"][off[1] + 1] = 5
    gpu, ref = run_multi(case), oracle.accept(case, test=2)
    for k in ("status", "accepted_len", "bonus_token", "path"):
        assert np.array_equal(gpu[k], ref[k]), k


@pytest.mark.parametrize("num", [2, 4])
def test_logits_decisions_away_from_ties(num):
    case = wl.make_case(wl.config(num), parts=("accept",), kind="logits")
    gpu, ref = run_multi(case), oracle.accept(case, test=2)
    off = case["node_offsets"]
    u = case["uniforms"].astype(np.float64)
    rp = ref["pq"].astype(np.float64)
    gap = np.abs(u * rp[:, 1] - rp[:, 0])
    near = gap <= 64 * PQ_RTOL * np.maximum(np.abs(rp[:, 0]), 1e-30)
    mismatched = 0
    for b in range(case["batch"]):
        same = (gpu["accepted_len"][b] == ref["accepted_len"][b] and
                np.array_equal(gpu["path"][b], ref["path"][b]))
        if not same:
            mismatched += 1
            assert near[off[b]:off[b + 1]].any(), f"tree {b} differs without a near-tie"
    assert mismatched <= max(1, case["batch"] // 8)
