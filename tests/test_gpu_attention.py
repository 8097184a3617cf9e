"""GPU parity of tv_tree_attention (through the C ABI) against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation), asserted on the fp32 output of
every comparison by tv_testlib.assert_attention_close: max-abs error <= 1e-2
over all elements, |g - r| <= 1e-2 + 2e-2*|r| element by element, and every
output row (one node, one head) within 2e-2 of its largest magnitude.  The
element-wise relative error over elements with |r| >= 1e-2 is reported
($TV_PARITY_LOG), not asserted (P is rounded to bf16 before P.V).  The bf16
output of the same inputs must be the fp32 output rounded to nearest even,
bit for bit.

Full sizes: every element of the 7B-like, serving and multimodal workloads;
on the long-context workload every row of one KV head of one sequence (all
m-tiles and every prefix split) plus a random sample of the rest.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import (assert_attention_close, assert_bf16_is_rounded_fp32, gather_rows,
                        run_attention, sample_rows)

pytestmark = pytest.mark.gpu


def full_compare(case, what, **kw):
    gpu, status = run_attention(case, **kw)
    assert np.all(status == 0), status
    ref = oracle.tree_attention(case)
    res = assert_attention_close(gpu, ref, what)
    assert np.all(assert_bf16_is_rounded_fp32(case, gpu, what, **kw) == 0)
    return res


# ---------------------------------------------------------------- small shapes
def test_tiny_config_full():
    case = wl.make_case(wl.config(1), parts=("attn",))
    full_compare(case, "tiny")


@pytest.mark.parametrize("d", [64, 128])
def test_single_tile_chain(d):
    cfg = wl.config(2, hq=2, hkv=2, d=d, prefix=(64, 64), n=(1, 1), batch=1)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, f"one tile d={d}")


def test_7b_shape_reduced_heads():
    cfg = wl.config(2, hq=8, hkv=8)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "7b-like, 8 heads")


def test_serving_shape_ragged_paged_gqa():
    cfg = wl.config(3, batch=5, hq=8, hkv=2, prefix=(0, 700), n=(1, 70), depth=6)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "serving reduced")


def test_multimodal_shape_group7():
    cfg = wl.config(4, batch=2, hq=7, hkv=1, prefix=(600, 600), image_tokens=200, vocab=3000)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "multimodal reduced (g=7, 128 nodes)")


def test_long_shape_split_kv_and_four_node_tiles():
    cfg = wl.config(5, batch=1, hq=16, hkv=2, prefix=(5000, 5000), vocab=2000)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "long reduced (splits, 256 nodes)")


def test_head_dim_64_gqa_ragged():
    cfg = wl.config(3, batch=3, hq=12, hkv=3, d=64, prefix=(1, 300), n=(2, 40), shuffle=True)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "d=64")


def test_empty_prefix_and_root_only_trees():
    cfg = wl.config(3, batch=4, hq=4, hkv=1, prefix=(0, 0), n=(1, 3))
    cfg["prefix_lens"] = [0, 0, 5, 17]
    cfg["nodes"] = [1, 3, 1, 2]
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "empty prefix / N=1")


def test_stale_page_tails_do_not_leak():
    """Pool slots past a sequence's end hold NaN: they must not reach the output."""
    cfg = wl.config(3, batch=3, hq=4, hkv=2, prefix=(30, 30), n=(5, 9))
    cfg["prefix_lens"] = [7, 30, 45]
    case = wl.make_case(cfg, parts=("attn",))
    nan_bf16 = np.uint16(0x7FC0)
    for b, L in enumerate(case["prefix_lens"]):
        for t in range(L, ((L + 63) // 64) * 64):
            if t // 16 < case["block_table"].shape[1] and t // 16 < (L + 15) // 16:
                pg = case["block_table"][b, t // 16]
                case["k_prefix"][pg, :, t % 16] = nan_bf16
                case["v_prefix"][pg, :, t % 16] = nan_bf16
    full_compare(case, "NaN page tails")


def test_many_sequences_many_splits():
    cfg = wl.config(3, batch=2, hq=2, hkv=1, prefix=(3000, 9000), n=(3, 20))
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "split-kv varlen")


@pytest.mark.parametrize("batch", [256, 300])
def test_batch_at_and_past_the_ordering_limit(batch):
    # up to 256 sequences the CTAs take the sequences longest first; past
    # that they take them in batch order
    cfg = wl.config(3, batch=batch, hq=2, hkv=1, prefix=(0, 300), n=(1, 6))
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, f"batch {batch}")


def test_many_tiny_sequences_take_several_scheduling_rounds():
    """2048 sequences of 1..3 nodes without a prefix on 4 KV heads: each CTA
    gets more pieces than one scheduling round holds (32), so it rebuilds its
    piece list several times."""
    cfg = wl.config(3, batch=2048, hq=4, hkv=4, d=64, prefix=(0, 0), n=(1, 3))
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "2048 tiny sequences")


def test_max_nodes_512_chain():
    cfg = wl.config(2, batch=1, hq=2, hkv=2, d=64, prefix=(40, 40))
    cfg["parent"] = [[-1] + list(range(511))]
    cfg["nodes"] = [512]
    cfg["n"] = (512, 512)
    case = wl.make_case(cfg, parts=("attn",))
    full_compare(case, "512-node chain", max_nodes=512)


def test_bad_tree_and_bad_block_report_status_and_zero_output():
    cfg = wl.config(3, batch=3, hq=4, hkv=2, prefix=(40, 40), n=(4, 4))
    case = wl.make_case(cfg, parts=("attn",))
    off = case["node_offsets"]
    case["parent"][off[1] + 2] = 3          # parent not before the node
    case["block_table"][2, 1] = 10 ** 6     # block id out of range
    gpu, status = run_attention(case)
    assert list(status) == [0, 5, 5]
    assert np.all(gpu[off[1]:off[3]] == 0)
    assert list(assert_bf16_is_rounded_fp32(case, gpu, "bad tree")) == [0, 5, 5]
    ref = oracle.tree_attention_rows(case, [(0, i, h) for i in range(4) for h in range(4)])
    assert_attention_close(gpu[off[0]:off[1]].reshape(-1, case["head_dim"]), ref, "good sequence")


def test_repeatable_bitwise():
    """Split units merge their pieces in a fixed order: repeated calls agree
    bit for bit (here every unit is split over several CTAs)."""
    case = wl.make_case(wl.config(3, batch=3, hq=8, hkv=2, prefix=(100, 900)), parts=("attn",))
    a, _ = run_attention(case)
    b, _ = run_attention(case)
    assert np.array_equal(a, b)


def test_malformed_sequences_with_prefix_splits_are_zeroed():
    """Long prefixes (several splits per tile): a bad parent, an out-of-range
    block id and a prefix longer than max_prefix_len each give status 5 and an
    all-zero output for that sequence; the others stay exact."""
    cfg = wl.config(3, batch=5, hq=8, hkv=2, prefix=(1900, 2040), n=(6, 12), shuffle=True)
    case = wl.make_case(cfg, parts=("attn",))
    off = case["node_offsets"]
    case["parent"][off[1] + 3] = 4                      # parent after the node
    case["block_table"][2, 60] = -7                      # block id out of range, mid-prefix
    lens = case["prefix_lens"].copy()
    lens[3] = 2100                                       # longer than the host hint below
    case["prefix_lens"] = lens
    nblk = (2100 + 15) // 16
    if case["block_table"].shape[1] < nblk:
        extra = np.zeros((case["batch"], nblk - case["block_table"].shape[1]), np.int32)
        case["block_table"] = np.concatenate([case["block_table"], extra], 1)
    gpu, status = run_attention(case, max_prefix_len=2048)
    assert list(status) == [0, 5, 5, 5, 0], status
    assert list(assert_bf16_is_rounded_fp32(case, gpu, "malformed", max_prefix_len=2048)) == \
        [0, 5, 5, 5, 0]
    for b in (1, 2, 3):
        assert np.all(gpu[off[b]:off[b + 1]] == 0), b
    rows = [(b, i, h) for b in (0, 4) for i in range(off[b + 1] - off[b]) for h in range(8)]
    ref = oracle.tree_attention_rows(case, rows)
    got = np.concatenate([gpu[off[b]:off[b + 1]].reshape(-1, case["head_dim"]) for b in (0, 4)])
    assert_attention_close(got, ref, "good sequences next to malformed split ones")


# ---------------------------------------------------------------- full sizes
@pytest.mark.parametrize("num", [2, 3, 4])
def test_full_size_config_every_element(num):
    case = wl.make_case(wl.config(num), parts=("attn",))
    gpu, status = run_attention(case)
    assert np.all(status == 0)
    ref = oracle.tree_attention(case)
    assert_attention_close(gpu, ref, f"config {num} every element")
    assert np.all(assert_bf16_is_rounded_fp32(case, gpu, f"config {num}") == 0)


def test_long_context_one_kv_head_every_row_plus_sample():
    """Long context: all 2048 packed rows (256 nodes x 8 query heads) of KV
    head 3 of sequence 1, which span every m-tile and every prefix split, and a
    random sample of rows of every sequence."""
    case = wl.make_case(wl.config(5), parts=("attn",))
    gpu, status = run_attention(case)
    assert np.all(status == 0)
    assert np.all(np.isfinite(gpu))
    g = case["num_q_heads"] // case["num_kv_heads"]
    kvh, b = 3, 1
    N = int(case["node_offsets"][b + 1] - case["node_offsets"][b])
    head_rows = np.asarray([(b, i, kvh * g + h) for i in range(N) for h in range(g)], np.int32)
    rows = np.concatenate([head_rows, sample_rows(case, 48, seed=5)])
    ref = oracle.tree_attention_rows(case, rows)
    assert_attention_close(gather_rows(gpu, case, rows), ref, "config 5 one kv head + sample")


@pytest.mark.parametrize("num", [2, 3, 4, 5])
def test_full_size_config_sampled_rows(num):
    case = wl.make_case(wl.config(num), parts=("attn",))
    gpu, status = run_attention(case)
    assert np.all(status == 0)
    assert np.all(np.isfinite(gpu))
    rows = sample_rows(case, 48, seed=num)
    ref = oracle.tree_attention_rows(case, rows)
    assert_attention_close(gather_rows(gpu, case, rows), ref, f"config {num} sampled rows")
