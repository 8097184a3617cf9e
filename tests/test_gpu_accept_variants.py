"""GPU parity of the accept-test variants against the oracle: the ratio test
with per-sequence calibration factors is bit-exact; the log-space clamped
test (fp32 log/exp on both sides, from different math libraries) must agree
on every tree that has no node within 1e-5 of its acceptance boundary."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import accept_device, ensure_built

pytestmark = pytest.mark.gpu

CASES = [(1, {}), (2, {}), (3, dict(batch=8, n=(10, 60))), (5, dict(batch=2, vocab=20000))]


def _gpu(case, **kw):
    ensure_built()
    t = accept_device(case)
    g = kw.pop("gamma", None)
    if g is not None:
        kw["gamma"] = torch.from_numpy(np.ascontiguousarray(g, np.float32)).cuda()
    r = tv.accept(t["target"], t["draft"], t["tokens"], t["parent"], t["off"], t["uniforms"],
                  t["mask"], max_nodes=int(case["max_nodes"]), kind="probs", debug_pq=True, **kw)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.cpu().numpy()) for k, v in r.items()}


@pytest.mark.parametrize("num, over", CASES)
def test_gamma_ratio_test_bit_exact(num, over):
    case = wl.make_case(wl.config(num, **over), parts=("accept",), kind="probs")
    gamma = np.random.default_rng(num).uniform(0.3, 3.0, case["batch"]).astype(np.float32)
    g = _gpu(case, gamma=gamma)
    r = oracle.accept(case, gamma=gamma)
    for k in ("accepted_len", "path", "bonus_token", "status"):
        assert np.array_equal(g[k], r[k]), k
    assert np.array_equal(g["debug_pq"], r["pq"])


@pytest.mark.parametrize("num, over", CASES)
@pytest.mark.parametrize("clamp", [20.0, 2.0])
def test_log_clamp_test_matches_away_from_the_boundary(num, over, clamp):
    case = wl.make_case(wl.config(num, **over), parts=("accept",), kind="probs")
    gamma = np.random.default_rng(num + 7).uniform(0.5, 2.0, case["batch"]).astype(np.float32)
    g = _gpu(case, test="log_clamp", log_clamp=clamp, gamma=gamma)
    r = oracle.accept(case, test=1, log_clamp=clamp, gamma=gamma)
    pq = r["pq"].astype(np.float64)
    off = case["node_offsets"]
    u = case["uniforms"].astype(np.float64)
    checked = 0
    for b in range(case["batch"]):
        sl = slice(off[b] + 1, off[b + 1])
        with np.errstate(divide="ignore", invalid="ignore"):
            rr = np.clip(np.log(pq[sl, 0]) - np.log(pq[sl, 1]) + np.log(float(gamma[b])), -clamp, clamp)
        prob = np.where(rr >= 0, 1.0, np.exp(rr))
        if np.any(np.abs(u[sl] - prob) < 1e-5):
            continue
        checked += 1
        for k in ("accepted_len", "path", "bonus_token", "status"):
            assert np.array_equal(g[k][b], r[k][b]), (k, b)
    assert checked >= 1


def test_bad_gamma_marks_the_tree():
    case = wl.make_case(wl.config(3, batch=4, vocab=500, n=(5, 9)), parts=("accept",), kind="probs")
    gamma = np.array([1.0, 0.0, np.nan, 2.0], np.float32)
    g = _gpu(case, gamma=gamma)
    r = oracle.accept(case, gamma=gamma)
    assert list(g["status"]) == [0, 5, 5, 0] == list(r["status"])
    assert np.array_equal(g["accepted_len"], r["accepted_len"])
