"""The C-ABI library builds, loads and exports every entry point that
include/tv.h declares; host-side argument checks reject bad calls before any
device work (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tv.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tv_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tv_tree_attention", "tv_accept", "tv_tree_attention_workspace_size",
              "tv_accept_workspace_size", "tv_status_string", "tv_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(tv.EXPORTS) <= set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.tv_version() == 100
    assert tv.status_string(0) == "TV_OK"
    assert tv.status_string(5) == "TV_ERR_BAD_TREE"
    assert tv.status_string(99) == "TV_ERR_UNKNOWN"


def _params(**kw):
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                max_blocks_per_seq=8, num_blocks=16, max_nodes=64, total_nodes=100,
                max_prefix_len=128, softmax_scale=0.0, out_dtype=0)
    base.update(kw)
    return tv.AttnParams(**base)


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(num_q_heads=7), dict(block_size=32),
                                 dict(max_nodes=513), dict(max_nodes=0), dict(batch=0),
                                 dict(max_prefix_len=1000), dict(total_nodes=1),
                                 dict(out_dtype=2)])
def test_attention_argument_errors_before_launch(lib, bad):
    p = _params(**bad)
    dummy = C.c_void_p(4096)  # never dereferenced: the call fails on the host
    rc = lib.tv_tree_attention(C.byref(p), *([dummy] * 11), None, C.c_size_t(0), None)
    assert rc in (tv.TV_ERR_INVALID_ARG, tv.TV_ERR_UNSUPPORTED)


def test_attention_null_pointer_rejected(lib):
    p = _params()
    dummy = C.c_void_p(4096)
    args = [dummy] * 11
    args[3] = None
    assert lib.tv_tree_attention(C.byref(p), *args, None, C.c_size_t(0), None) == tv.TV_ERR_INVALID_ARG
    args = [dummy] * 11
    args[0] = C.c_void_p(4097)  # misaligned
    assert lib.tv_tree_attention(C.byref(p), *args, None, C.c_size_t(0), None) == tv.TV_ERR_INVALID_ARG


def test_attention_workspace_size_rules(lib):
    assert lib.tv_tree_attention_workspace_size(C.byref(_params(head_dim=96))) == 0
    assert lib.tv_tree_attention_workspace_size(C.byref(_params(out_dtype=2))) == 0
    # two counters per CTA (rounded to 256 bytes), then two slots per CTA of
    # 256 rows x D fp32, 256 (m, l) pairs and a 256-byte flag area
    for d in (64, 128):
        plan = tv.attention_plan(_params(head_dim=d), sms=152)
        ctas = plan["ctas"]
        slot = 256 * d * 4 + 256 * 8 + 256
        assert plan["workspace_bytes"] == (ctas * 8 + 255) // 256 * 256 + 2 * ctas * slot


def test_attention_refuses_a_short_workspace(lib):
    p = _params()
    dummy = C.c_void_p(4096)
    need = lib.tv_tree_attention_workspace_size(C.byref(p))
    assert need > 0
    assert lib.tv_tree_attention(C.byref(p), *([dummy] * 11), None, C.c_size_t(0), None) == \
        tv.TV_ERR_WORKSPACE
    assert lib.tv_tree_attention(C.byref(p), *([dummy] * 11), dummy, C.c_size_t(need - 16),
                                 None) == tv.TV_ERR_WORKSPACE


@pytest.mark.parametrize("bad", [dict(vocab=0), dict(vocab=1 << 18), dict(max_nodes=600),
                                 dict(kind=3), dict(batch=0), dict(total_nodes=0)])
def test_accept_argument_errors_before_launch(lib, bad):
    base = dict(batch=2, vocab=1000, max_nodes=16, total_nodes=20, kind=0)
    base.update(bad)
    p = tv.AcceptParams(**base)
    dummy = C.c_void_p(4096)
    args = [dummy] * 12
    args[6] = None  # retained_mask optional
    args[11] = None  # debug_pq optional
    assert lib.tv_accept(C.byref(p), *args, None, C.c_size_t(0), None) == tv.TV_ERR_INVALID_ARG


def test_accept_workspace_size_rules(lib):
    # per (row, 8192-entry vocabulary chunk): a float2 and a uint64
    p = tv.AcceptParams(batch=2, vocab=20000, max_nodes=16, total_nodes=20, kind=1)
    assert lib.tv_accept_workspace_size(C.byref(p)) == 20 * 3 * 16
    p = tv.AcceptParams(batch=2, vocab=1 << 18, max_nodes=16, total_nodes=20, kind=1)
    assert lib.tv_accept_workspace_size(C.byref(p)) == 0


def test_accept_logits_without_workspace_is_refused(lib):
    p = tv.AcceptParams(batch=2, vocab=1000, max_nodes=16, total_nodes=20, kind=1)
    dummy = C.c_void_p(4096)
    args = [dummy] * 12
    args[6] = None
    args[11] = None
    assert lib.tv_accept(C.byref(p), *args, None, C.c_size_t(0), None) == tv.TV_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(OSError):
        tv.load(str(tmp_path / "missing_libtv.so"))


@pytest.mark.parametrize("bad", [dict(rows=0), dict(vocab=0), dict(vocab=(1 << 18) + 1),
                                 dict(mass=0.0), dict(mass=float("nan")), dict(mass=33.0),
                                 dict(mass=1e-13)])
def test_retained_set_argument_errors_before_launch(lib, bad):
    base = dict(rows=4, vocab=1000, mass=0.7)
    base.update(bad)
    p = tv.RetainParams(**base)
    dummy = C.c_void_p(4096)
    assert lib.tv_retained_set(C.byref(p), dummy, dummy, None, None, None, None) == \
        tv.TV_ERR_INVALID_ARG


def test_commit_argument_errors_before_launch(lib):
    dummy = C.c_void_p(4096)
    args = [dummy] * 12
    ok = dict(batch=2, num_kv_heads=2, head_dim=128, block_size=16, max_blocks_per_seq=8,
              num_blocks=16, max_nodes=16, total_nodes=20)
    for bad in (dict(batch=0), dict(block_size=8), dict(max_nodes=600), dict(total_nodes=1)):
        p = tv.CommitParams(**dict(ok, **bad))
        assert lib.tv_commit_kv(C.byref(p), *args, None) == tv.TV_ERR_INVALID_ARG
    p = tv.CommitParams(**dict(ok, head_dim=96))
    assert lib.tv_commit_kv(C.byref(p), *args, None) == tv.TV_ERR_UNSUPPORTED
    # new_prefix_lens aliasing prefix_lens is refused
    p = tv.CommitParams(**ok)
    aliased = list(args)
    aliased[7] = C.c_void_p(8192)
    aliased[10] = C.c_void_p(8192)
    assert lib.tv_commit_kv(C.byref(p), *aliased, None) == tv.TV_ERR_INVALID_ARG
    assert tv.status_string(tv.TV_ERR_NO_PAGE) == "TV_ERR_NO_PAGE"


@pytest.mark.parametrize("bad", [dict(test=3), dict(test=-1), dict(log_clamp=-1.0), dict(log_clamp=100.0),
                                 dict(log_clamp=float("nan"))])
def test_accept_options_checked_before_launch(lib, bad):
    p = tv.AcceptParams(batch=2, vocab=1000, max_nodes=16, total_nodes=20, kind=0)
    o = tv.AcceptOptions(**dict(dict(test=0, log_clamp=0.0, gamma=None), **bad))
    dummy = C.c_void_p(4096)
    args = [dummy] * 12
    args[6] = None
    args[11] = None
    assert lib.tv_accept_ex(C.byref(p), C.byref(o), *args, None, C.c_size_t(0), None) == \
        tv.TV_ERR_INVALID_ARG


@pytest.mark.parametrize("limit_ns", [0, 999_999, 1_000_000_001])
def test_selftest_wait_timeout_checks_arguments(lib, limit_ns):
    dummy = C.c_void_p(4096)
    assert lib.tv_selftest_wait_timeout(dummy, dummy, C.c_ulonglong(limit_ns), None) == \
        tv.TV_ERR_INVALID_ARG
    assert lib.tv_selftest_wait_timeout(None, dummy, C.c_ulonglong(10_000_000), None) == \
        tv.TV_ERR_INVALID_ARG


def _plan(batch, hq, hkv, d, max_nodes, max_prefix):
    blocks = (max_prefix + 15) // 16
    return tv.AttnParams(batch, hq, hkv, d, 16, max(1, blocks), max(1, batch * blocks), max_nodes,
                         batch * max_nodes, max_prefix, 0.0, 0)


# (lanes, virtual CTAs) on 152 SMs: lanes = m-tile pairs of the largest tree
# (256 packed rows each), virtual CTAs = 152 // lanes, fewer when the line of
# key tiles (batch x Hkv x layers x (prefix tiles + node tiles)) gives fewer
# than 3 tiles each
@pytest.mark.parametrize("shape, lanes, vctas", [
    ((1, 4, 4, 64, 15, 128), 1, 2),          # tiny: 4 heads x 2 tiles = 8 tiles
    ((1, 32, 32, 128, 64, 1024), 1, 96),     # 7B-like: 32 x 9 = 288 tiles
    ((16, 32, 8, 128, 64, 3959), 1, 152),    # serving: 16 x 8 x 32 tiles
    ((4, 28, 4, 128, 128, 1600), 4, 38),     # multimodal: 896 rows = 4 pairs, 224 tiles
    ((4, 64, 8, 128, 256, 32768), 8, 19),    # long: 2048 rows = 8 pairs, 8256 tiles
    ((1, 64, 8, 128, 256, 32768), 8, 19),    # long, one sequence
])
def test_launch_plan(lib, shape, lanes, vctas):
    plan = tv.attention_plan(_plan(*shape), sms=152)
    assert (plan["lanes"], plan["virtual_ctas"]) == (lanes, vctas)
    assert plan["ctas"] == lanes * vctas <= 152 and plan["min_tiles"] == 3
    # the fixed scratch array of the no-allocation entry point holds every plan
    assert plan["workspace_bytes"] <= 64 << 20


def test_launch_plan_scales_with_the_sm_count(lib):
    p = _plan(16, 32, 8, 128, 64, 3959)
    for sms in (1, 76, 148, 160):
        plan = tv.attention_plan(p, sms=sms)
        assert plan["ctas"] == sms


def test_launch_plan_rejects_invalid_params(lib):
    for p in (_plan(1, 6, 4, 128, 64, 1024), _plan(1, 4, 4, 96, 64, 1024)):
        with pytest.raises(tv.TVError):
            tv.attention_plan(p, sms=152)
