"""GPU parity of tv_retained_set against the oracle's retained set: masks,
exact fixed-point mass Z, its fp32 value and the kept counts must match bit
for bit on every row (every decision is an exact integer comparison)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import ensure_built

pytestmark = pytest.mark.gpu


def _run(rows, mass):
    ensure_built()
    q = torch.from_numpy(np.ascontiguousarray(rows, np.float32)).cuda()
    m, zf, z, k = tv.retained_set(q, mass)
    torch.cuda.synchronize()
    return (m.cpu().numpy().view(np.uint32), zf.cpu().numpy().view(np.uint64), z.cpu().numpy(),
            k.cpu().numpy())


def _check(rows, mass):
    got = _run(rows, mass)
    ref = oracle.retained_set(rows, mass)
    for name, g, r in zip(("mask", "z_fixed", "z", "kept"), got, ref):
        assert np.array_equal(g, r), (name, np.nonzero(np.any(np.atleast_2d(g != r), axis=-1)))
    return got


@pytest.mark.parametrize("num", [2, 4, 5])
def test_workload_draft_rows(num):
    case = wl.make_case(wl.config(num, batch=1, n=(24, 24), depth=3), parts=("accept",))
    got = _check(case["draft_probs"], 0.7)
    if num == 4:  # the multimodal workload's own masks come from the fp64 recipe
        assert np.array_equal(got[0], case["retained_mask"])


@pytest.mark.parametrize("V", [1, 31, 33, 1000, 16384, 16385, 40003, 1 << 18])
@pytest.mark.parametrize("mass", [1e-6, 0.3, 0.7, 1.0, 2.0])
def test_sizes_and_masses(V, mass):
    g = np.random.default_rng(V)
    logits = g.standard_normal((3, V)) * 2.0
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    rows = (p / p.sum(axis=1, keepdims=True)).astype(np.float32)
    _check(rows, mass)


def test_ties_zeros_nans_and_negatives():
    V = 20000
    g = np.random.default_rng(5)
    rows = np.zeros((6, V), np.float32)
    rows[0] = np.float32(1.0 / V)                              # all tied
    rows[1] = g.choice([0.0, 1e-5, 2e-5, 5e-5], size=V).astype(np.float32)  # few values
    rows[2] = 0.0                                              # no mass at all
    rows[3] = g.random(V).astype(np.float32) / V * 2
    rows[3, g.integers(0, V, 50)] = np.nan                     # NaN counts as 0
    rows[3, g.integers(0, V, 50)] = -1.0                       # negatives count as 0
    rows[4] = np.float32(1e-13)                                # below the 2^-40 quantum
    rows[5, 17] = 1.0                                          # a single token
    _check(rows, 0.7)
    _check(rows, 0.999)


def test_many_rows():
    g = np.random.default_rng(11)
    logits = g.standard_normal((300, 4099)) * 3.0
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    _check((p / p.sum(axis=1, keepdims=True)).astype(np.float32), 0.7)


def test_flat_rows_overflow_the_key_copy():
    """Rows whose crossing top-byte bucket holds more keys than shared memory
    keeps (the later passes read the row again): all tied, and mostly tied."""
    V = 1 << 18
    g = np.random.default_rng(21)
    rows = np.zeros((3, V), np.float32)
    rows[0] = np.float32(1.0 / V)
    rows[1] = np.float32(1.0 / V)
    rows[1, g.integers(0, V, 3000)] = np.float32(3.0 / V)
    rows[2] = (np.float32(1.0 / V) * (1.0 + 0.9 * g.random(V))).astype(np.float32)
    _check(rows, 0.7)
    _check(rows, 0.31)


def test_values_above_128():
    """Unnormalised rows with values >= 2^7 (top bytes above the 24 private
    buckets; weights clamped at 32)."""
    g = np.random.default_rng(22)
    V = 5000
    rows = (g.random((4, V)) * 1e-3).astype(np.float32)
    rows[0, g.integers(0, V, 5)] = np.float32(200.0)
    rows[1, :40] = (g.random(40) * 1e4 + 128.0).astype(np.float32)
    rows[2, 7] = np.float32(np.inf)
    rows[3, 100:110] = np.float32(31.5)
    for mass in (0.5, 20.0, 32.0):
        _check(rows, mass)
