"""Host-side logic of bench.py: the roofline bound choice, the algorithmic
byte and FLOP counts on a hand-sized tree, and the reference arm's JSON line
(the oracle on the host cores; no GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _chain_case():
    # one sequence, a 4-node chain (depths 0..3), prefix of 32 keys, g = 2
    return dict(num_q_heads=2, num_kv_heads=1, head_dim=64, prefix_lens=[32],
                node_offsets=[0, 4], parent=[-1, 0, 1, 2], batch=1)


def test_attention_counts_on_a_chain():
    c = _chain_case()
    # prefix K+V once (2 tensors x 2 bytes), Q + output (2 x 2 bytes), tree K+V
    assert bench.attention_bytes(c) == 4 * 32 * 64 + 4 * 4 * 2 * 64 + 4 * 4 * 64
    # 2 FLOPs per multiply-add in Q.K and P.V: every node sees 32 prefix keys
    # and depth+1 tree keys, 1+2+3+4 = 10 tree keys in all
    assert bench.attention_flops(c) == 4 * 4 * 32 * 64 * 2 + 4 * 64 * 2 * 10


def test_roofline_bound_follows_intensity():
    bw, tf = 6000.0, 1800.0  # ridge = 300 FLOP/B
    low = bench.roofline_entry(1e9, 100e9, 1e-3, bw, tf, "measured")
    assert low["bound"] == "hbm" and low["unit"] == "GB/s"
    assert low["achieved"] == pytest.approx(1000.0) and low["frac"] == pytest.approx(1000.0 / bw)
    high = bench.roofline_entry(1e9, 400e9, 1e-3, bw, tf, "measured")
    assert high["bound"] == "tensor" and high["unit"] == "TFLOP/s"
    assert high["achieved"] == pytest.approx(400.0) and high["frac"] == pytest.approx(400.0 / tf)
    assert "fallback" in bench.roofline_entry(1, 1, 1, bw, tf, "fallback")["peak_source"]


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"].startswith("tiny")
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data"):
        assert k in line


def test_percentiles_in_microseconds():
    p = bench.pct([0.001 * k for k in range(1, 102)])  # 1 .. 101 us, given in ms
    assert p["p50"] == pytest.approx(51.0)
    assert p["p10"] == pytest.approx(11.0) and p["p90"] == pytest.approx(91.0)
