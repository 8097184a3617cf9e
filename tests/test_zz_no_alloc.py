"""tv_tree_attention_no_alloc: tree attention for callers that cannot allocate
device memory (no workspace argument; the library keeps split-KV partials in
its own fixed device array).  Its output must match tv_tree_attention's on
the same inputs, on two calls in a row (the array keeps the previous call's
contents), and requests larger than the array must be refused on the host.

This file is collected last on purpose, so a stop-at-first-failure run has
already run every other test before this one."""
import ctypes as C

import numpy as np
import pytest
import torch

import speculative_decoding_tree_attention_gb300 as tv
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import ATOL, RTOL, attn_device, attention_errors, ensure_built

pytestmark = pytest.mark.gpu


def _call_no_alloc(lib, prm, t, out, status):
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda x: C.c_void_p(x.data_ptr())
    return lib.tv_tree_attention_no_alloc(C.byref(prm), p(t["q"]), p(t["kp"]), p(t["vp"]),
                                          p(t["table"]), p(t["kn"]), p(t["vn"]), p(t["parent"]),
                                          p(t["lens"]), p(t["off"]), p(out), p(status), stream)


@pytest.mark.parametrize("num, overrides", [
    (2, {}),                                                      # 7B-like: two prefix splits
    (3, dict(batch=6, hq=8, hkv=2, prefix=(300, 3000), n=(5, 64))),  # ragged, several splits
])
def test_no_alloc_matches_workspace_entry_point_twice(num, overrides):
    lib = ensure_built()
    case = wl.make_case(wl.config(num, **overrides), parts=("attn",))
    t = attn_device(case)
    max_nodes = int(case["max_nodes"])
    mpl = int(max(1, int(np.max(case["prefix_lens"]))))
    ref_out, ref_status = tv.tree_attention(t["q"], t["kp"], t["vp"], t["table"], t["kn"],
                                            t["vn"], t["parent"], t["lens"], t["off"],
                                            max_nodes=max_nodes, max_prefix_len=mpl)
    prm = tv.attention_params(t["q"], t["kp"], t["table"], t["lens"],
                              num_kv_heads=case["num_kv_heads"], max_nodes=max_nodes,
                              max_prefix_len=mpl)
    assert 0 < tv.attention_workspace_size(prm) <= lib_scratch_bytes()
    ref = ref_out.float().cpu().numpy()
    for call in range(2):
        out = torch.full_like(t["q"], float("nan"))
        status = torch.full((case["batch"],), -1, dtype=torch.int32, device=t["q"].device)
        assert _call_no_alloc(lib, prm, t, out, status) == tv.TV_OK
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.array_equal(status.cpu().numpy(), ref_status.cpu().numpy())
        assert np.all(np.isfinite(got))
        max_abs, row_rel, ratio = attention_errors(got, ref)
        assert ratio <= 1.0 and row_rel <= RTOL, (call, max_abs, row_rel)


def lib_scratch_bytes():
    return 32 << 20  # TV_NO_ALLOC_SCRATCH_BYTES


def test_no_alloc_refuses_requests_beyond_the_array():
    lib = ensure_built()
    # serving-batch shapes: 16 sequences x 8 KV heads x 2 m-tiles, long prefixes
    # split in two -> about 34 MB of partials on a 152-SM GPU
    candidates = [dict(batch=b, num_q_heads=32, num_kv_heads=8, max_nodes=64) for b in (16, 12, 8)]
    prm = None
    for c in candidates:
        p = tv.AttnParams(head_dim=128, block_size=16, max_blocks_per_seq=256,
                          num_blocks=c["batch"] * 256, total_nodes=c["batch"] * 64,
                          max_prefix_len=4096, softmax_scale=0.0, **c)
        if tv.attention_workspace_size(p) > lib_scratch_bytes():
            prm = p
            break
    assert prm is not None, "no candidate plan exceeds the scratch array on this GPU"
    dummy = C.c_void_p(4096)  # never dereferenced: refused on the host
    rc = lib.tv_tree_attention_no_alloc(C.byref(prm), *([dummy] * 11), None)
    assert rc == tv.TV_ERR_WORKSPACE
