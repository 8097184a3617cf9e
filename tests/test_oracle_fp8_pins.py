"""Pins of the oracle's E4M3 input path (CPU only): the FP8 form of the
attention inputs, E4M3 codes with one fp32 scale per row of D elements.

- The oracle's decoding gives the format's textbook values (1, 1.5, 2, the
  largest normal 448, the smallest normal 2^-6 and subnormal 2^-9, signed
  zero, NaN at S.1111.111), is strictly increasing over the positive codes and
  odd in the sign bit.
- The input quantiser rounds to the nearest code (checked by brute force over
  all finite codes), ties to the even code, saturates at 448, and every
  finite code survives a decode / encode round trip.
- Attention on E4M3 inputs equals attention on the same values given as bf16
  (E4M3 values times powers of two are exact in bf16), so the fp8 path reuses
  the pinned fp64 attention with nothing lost or misplaced: a scale applied to
  the wrong row, or a wrong decode, changes the output."""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl


def test_decode_textbook_values():
    v = oracle.e4m3_value
    assert v(0x38) == 1.0 and v(0x3C) == 1.5 and v(0x40) == 2.0
    assert v(0x7E) == 448.0 and v(0x08) == 2.0 ** -6 and v(0x01) == 2.0 ** -9
    assert v(0x07) == 7 * 2.0 ** -9 and v(0x0F) == 1.875 * 2.0 ** -6
    assert v(0x00) == 0.0 and np.signbit(v(0x80)) and v(0x80) == 0.0
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0xB8) == -1.0 and v(0xFE) == -448.0


def test_decode_monotone_and_odd():
    pos = [oracle.e4m3_value(c) for c in range(127)]
    assert all(a < b for a, b in zip(pos, pos[1:]))
    for c in range(127):
        assert oracle.e4m3_value(c | 0x80) == -pos[c]


def test_encoder_nearest_ties_even_saturation():
    table = np.array([oracle.e4m3_value(c) for c in range(127)])
    g = wl.rng(5, 701)
    x = np.concatenate([g.normal(0, 30, 4000), g.uniform(-500, 500, 2000),
                        g.normal(0, 2.0 ** -7, 2000)])
    codes = wl.e4m3_encode(x)
    for xi, c in zip(x, codes):
        mag = min(abs(xi), 448.0)
        best = np.min(np.abs(table - mag))
        got = oracle.e4m3_value(int(c) & 0x7F)
        assert abs(got - mag) == best, (xi, c)
        assert (int(c) >> 7) == (1 if np.signbit(xi) else 0)
    # exact midpoints go to the even code
    for lo in range(126):
        mid = (table[lo] + table[lo + 1]) / 2
        assert int(wl.e4m3_encode(mid)) == (lo if lo % 2 == 0 else lo + 1)
    assert int(wl.e4m3_encode(1e6)) == 0x7E and int(wl.e4m3_encode(-1e6)) == 0xFE
    assert int(wl.e4m3_encode(np.nan)) == 0x7F


def test_every_finite_code_round_trips():
    for c in list(range(127)) + list(range(128, 255)):
        assert int(wl.e4m3_encode(oracle.e4m3_value(c))) == c


def _small_case(seed):
    cfg = wl.config(3, batch=3, hq=4, hkv=2, d=64, prefix=(20, 70), n=(3, 12), shuffle=True)
    cfg["seed"] = seed
    return wl.make_case(cfg, parts=("attn",))


@pytest.mark.parametrize("seed", [1, 2])
def test_e4m3_attention_equals_bf16_attention_on_equal_values(seed):
    base = _small_case(seed)
    g = wl.rng(seed, 702)
    fp8 = dict(base, dtype="e4m3")
    bf = dict(base)
    for k in ("q", "k_prefix", "v_prefix", "k_nodes", "v_nodes"):
        shape = base[k].shape
        # moderate magnitudes (exponent field <= 7: |value| < 2), so that no
        # softmax row is one-hot; random signs
        codes = ((g.integers(0, 2, size=shape) << 7) | (g.integers(0, 8, size=shape) << 3) |
                 g.integers(0, 8, size=shape)).astype(np.uint8)
        rows = int(np.prod(shape[:-1]))
        scale = (2.0 ** g.integers(-3, 4, size=rows)).astype(np.float32).reshape(shape[:-1])
        vals = np.vectorize(oracle.e4m3_value)(codes) * scale[..., None]
        fp8[k], fp8[k + "_scale"] = codes, scale
        bf[k] = wl.to_bf16_bits(vals)
        assert np.array_equal(wl.bf16_bits_to_f32(bf[k]).astype(np.float64), vals)  # exact
    a = oracle.tree_attention(fp8)
    b = oracle.tree_attention(bf)
    assert np.array_equal(a, b)
    # a changed scale on a row the first sequence reads is seen
    moved = dict(fp8)
    sc = fp8["v_prefix_scale"].copy()
    sc[int(base["block_table"][0, 0]), 0, 0] *= np.float32(2.0)
    moved["v_prefix_scale"] = sc
    assert not np.array_equal(oracle.tree_attention(moved), a)


def test_quantised_workload_stays_close_to_bf16():
    base = _small_case(3)
    q8 = wl.e4m3_case(base)
    a, b = oracle.tree_attention(q8), oracle.tree_attention(base)
    # E4M3 keeps 4 significant bits: a relative step of 2^-4 per element
    assert np.abs(a - b).max() < 0.15
    assert np.abs(a - b).mean() < 0.02
