"""GPU parity of tv_tree_attention_fp8 (E4M3 inputs with one fp32 scale per
row of 128 codes; [EC] §9.2) through the C ABI, against the oracle's E4M3
path (the codes decoded from the format's definition, times their scales,
attention in fp64).

The inputs are the bf16 workloads re-quantised per row (workloads.e4m3_case).
Tolerance: as for the bf16 path (tv_testlib.assert_attention_close on the
fp32 output: max-abs 1e-2, allclose 1e-2 + 2e-2|r|, each row within 2e-2 of
its largest magnitude); the bf16 output is the fp32 output rounded once."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import assert_attention_close, ensure_built, gather_rows, sample_rows

pytestmark = pytest.mark.gpu


def run_fp8(case, out_dtype="fp32", max_prefix_len=None):
    ensure_built()
    dev = "cuda"
    u8 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.uint8)).to(dev)
    f32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    i32 = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.int32)).to(dev)
    mpl = int(max_prefix_len or max(1, int(np.max(case["prefix_lens"]))))
    out, st = tv.tree_attention_fp8(
        u8(case["q"]), f32(case["q_scale"]), u8(case["k_prefix"]), f32(case["k_prefix_scale"]),
        u8(case["v_prefix"]), f32(case["v_prefix_scale"]), i32(case["block_table"]),
        u8(case["k_nodes"]), f32(case["k_nodes_scale"]), u8(case["v_nodes"]),
        f32(case["v_nodes_scale"]), i32(case["parent"]), i32(case["prefix_lens"]),
        i32(case["node_offsets"]), max_nodes=int(case["max_nodes"]), max_prefix_len=mpl,
        out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st.cpu().numpy()


def full_compare_fp8(case, what, **kw):
    gpu, st = run_fp8(case, **kw)
    assert np.all(st == 0), st
    ref = oracle.tree_attention(case)
    res = assert_attention_close(gpu, ref, what)
    g16, st16 = run_fp8(case, out_dtype="bf16", **kw)
    assert np.all(st16 == 0)
    assert np.array_equal(wl.to_bf16_bits(gpu), wl.to_bf16_bits(g16)), what
    return res


def fp8(cfg):
    return wl.e4m3_case(wl.make_case(cfg, parts=("attn",)))


def test_tiny_shape_d128():
    full_compare_fp8(fp8(wl.config(2, batch=1, hq=2, hkv=2, prefix=(100, 100), n=(9, 9))),
                     "fp8 small")


def test_ragged_paged_gqa():
    full_compare_fp8(fp8(wl.config(3, batch=5, hq=8, hkv=2, prefix=(0, 700), n=(1, 70), depth=6)),
                     "fp8 serving reduced")


def test_group7_and_image_prefix():
    full_compare_fp8(fp8(wl.config(4, batch=2, hq=7, hkv=1, prefix=(600, 600), image_tokens=200,
                                   vocab=3000)), "fp8 multimodal reduced")


def test_split_units_and_four_node_tiles():
    full_compare_fp8(fp8(wl.config(5, batch=1, hq=16, hkv=2, prefix=(5000, 5000), vocab=2000)),
                     "fp8 long reduced")


def test_stale_page_tails_hold_nan_codes():
    """Codes past a sequence's end are NaN (0x7F): they must not reach the output."""
    cfg = wl.config(3, batch=3, hq=4, hkv=2, prefix=(30, 30), n=(5, 9))
    cfg["prefix_lens"] = [7, 30, 45]
    case = fp8(cfg)
    for b, L in enumerate(case["prefix_lens"]):
        for t in range(L, ((L + 15) // 16) * 16):
            pg = case["block_table"][b, t // 16]
            case["k_prefix"][pg, :, t % 16] = 0x7F
            case["v_prefix"][pg, :, t % 16] = 0x7F
    full_compare_fp8(case, "fp8 NaN page tails")


def test_v_scales_across_decades():
    """V row scales set per sequence from 1e-3 to 5e3 times the quantiser's
    (dequantised V up to about 3e4, inside the fp16 range of the converted
    rows) and, in one sequence, spread per row over a decade each way: each
    sequence's output divided by its factor matches the oracle's divided by it."""
    case = fp8(wl.config(3, batch=4, hq=8, hkv=2, prefix=(200, 600), n=(10, 40)))
    fac = [1e-3, 1.0, 30.0, 5e3]
    off, L = case["node_offsets"], case["prefix_lens"]
    spread = 10.0 ** wl.rng(77, 1).uniform(-1.0, 1.0, size=case["v_prefix_scale"].shape[1:])
    seen = set()
    for b in range(4):
        pages = case["block_table"][b, : (int(L[b]) + 15) // 16]
        assert not seen.intersection(pages.tolist())
        seen.update(pages.tolist())
        for pg in pages:
            case["v_prefix_scale"][pg] *= np.float32(fac[b]) * (spread if b == 1 else 1.0)
        case["v_nodes_scale"][off[b]:off[b + 1]] *= np.float32(fac[b])
    gpu, st = run_fp8(case)
    assert np.all(st == 0), st
    ref = oracle.tree_attention(case)
    for b in range(4):
        sl = slice(off[b], off[b + 1])
        assert_attention_close(gpu[sl] / fac[b], ref[sl] / fac[b], f"fp8 V scale x{fac[b]:g}")


def test_bad_tree_status_and_zeros():
    case = fp8(wl.config(3, batch=3, hq=4, hkv=2, prefix=(40, 40), n=(4, 4)))
    off = case["node_offsets"]
    case["parent"][off[1] + 2] = 3
    gpu, st = run_fp8(case)
    assert list(st) == [0, 5, 0]
    assert np.all(gpu[off[1]:off[2]] == 0)


@pytest.mark.parametrize("num", [2, 3, 4])
def test_full_size_every_element(num):
    full_compare_fp8(fp8(wl.config(num)), f"fp8 config {num} every element")


def test_long_context_one_kv_head_and_sample():
    case = fp8(wl.config(5))
    gpu, st = run_fp8(case)
    assert np.all(st == 0)
    g = case["num_q_heads"] // case["num_kv_heads"]
    N = int(case["node_offsets"][2] - case["node_offsets"][1])
    rows = np.concatenate([np.asarray([(1, i, 2 * g + h) for i in range(N) for h in range(g)], np.int32),
                           sample_rows(case, 48, seed=55)])
    ref = oracle.tree_attention_rows(case, rows)
    assert_attention_close(gather_rows(gpu, case, rows), ref, "fp8 config 5 one kv head + sample")
