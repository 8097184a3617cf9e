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
    """The rows alone (up to half a wave of rows: two CTAs a row), then
    repeated past a full wave of SMs, so that every row is also computed by
    one CTA (the full waves) and the last copies again by two."""
    rows = np.ascontiguousarray(rows, np.float32)
    ref = oracle.retained_set(rows, mass)
    got = _run(rows, mass)
    for name, g, r in zip(("mask", "z_fixed", "z", "kept"), got, ref):
        assert np.array_equal(g, r), (name, np.nonzero(np.any(np.atleast_2d(g != r), axis=-1)))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    k = -(-sms // rows.shape[0]) + 1
    tiled = _run(np.concatenate([rows] * k), mass)
    for name, g, r in zip(("mask", "z_fixed", "z", "kept"), tiled, ref):
        want = np.concatenate([r] * k)
        assert np.array_equal(g, want), (name, "tiled", np.nonzero(np.any(np.atleast_2d(g != want), axis=-1)))
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
    """Rows whose crossing exponent field holds more keys than the id list
    keeps (the later digits and the mask come from passes over the row): all
    tied, and mostly tied.  (A row of 20000 equal values, whose 16-bit prefix
    overflows only the small list, is in the ties test.)"""
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
    """Unnormalised rows with values >= 32 (exponent fields 132 and up, whose
    weights are clamped to 32, counted in shared buckets) and +inf."""
    g = np.random.default_rng(22)
    V = 5000
    rows = (g.random((4, V)) * 1e-3).astype(np.float32)
    rows[0, g.integers(0, V, 5)] = np.float32(200.0)
    rows[1, :40] = (g.random(40) * 1e4 + 128.0).astype(np.float32)
    rows[2, 7] = np.float32(np.inf)
    rows[3, 100:110] = np.float32(31.5)
    for mass in (0.5, 20.0, 32.0):
        _check(rows, mass)


def test_ties_at_tau_ranked_by_id():
    """Rows whose crossing key is shared by more entries than the ties to
    keep: the kept ties are those of lowest id.  7, 300 and 1500 ties, alone
    at their 16-bit key prefix (ranked in the small list), and 5000 ties, more
    than the small list holds (ranked by the pass over the row)."""
    g = np.random.default_rng(23)
    V = 6000
    rows = (g.random((4, V)) * 1e-4).astype(np.float32)
    for r, n in enumerate((7, 300, 1500, 5000)):
        rows[r, g.choice(V, n, replace=False)] = np.float32(2e-4)
    for mass in (0.0005, 0.03, 0.2, 0.45):
        _check(rows, mass)


def test_small_list_neighbours_of_tau():
    """Keys sharing tau's 16-bit prefix on both sides of it: one field, a few
    hundred distinct keys within one 2^-7 relative step, and exact ties."""
    g = np.random.default_rng(24)
    V = 50000
    rows = (g.random((2, V)) * 1e-6).astype(np.float32)
    base = np.float32(1e-4).view(np.uint32) & np.uint32(0xffff8000)
    for r in range(2):
        idx = g.choice(V, 600, replace=False)
        bits_ = base + g.integers(0, 1 << 15, 600).astype(np.uint32) // (1 << (8 * r))
        rows[r, idx] = bits_.view(np.float32)
    for mass in (0.01, 0.03, 0.05):
        _check(rows, mass)


def test_full_size_multimodal_rows():
    """The multimodal workload's 512 draft rows of 151936 at mass 0.7, the
    launch the benchmark times (four waves of one-CTA rows), bit for bit;
    the workload's own masks come from the fp64 recipe."""
    case = wl.make_case(wl.config(4), parts=("accept",))
    got = _check(case["draft_probs"], float(wl.config(4)["mask_mass"]))
    assert np.array_equal(got[0], case["retained_mask"])
