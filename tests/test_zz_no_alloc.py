"""tv_tree_attention_no_alloc: tree attention for callers that cannot allocate
device memory (code under stream capture, an operator inside an engine that
owns all device memory, a service that allocates nothing after start-up).
It takes no workspace: the arrival counters and partial-result slots the
launch plan needs come from a fixed device array owned by the library.  Its
output must match tv_tree_attention's on the same inputs, on two calls in a
row (the second call finds the first one's contents in the array).

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
    (2, {}),                                                      # 7B-like: prefix splits
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
    # the plan splits units, so the calls use the array's counters and slots
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
        assert max_abs <= ATOL and ratio <= 1.0 and row_rel <= RTOL, (call, max_abs, row_rel)


def lib_scratch_bytes():
    return 64 << 20  # TV_NO_ALLOC_SCRATCH_BYTES


def test_no_alloc_plans_fit_the_array():
    # every workload's plan on this device fits the array; a device with more
    # than 251 SMs would need more at D = 128 and be refused (TV_ERR_WORKSPACE)
    for b, hq, hkv, n, L in ((16, 32, 8, 64, 4096), (4, 64, 8, 256, 32768), (4, 28, 4, 128, 1600)):
        p = tv.AttnParams(batch=b, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=16,
                          max_blocks_per_seq=L // 16, num_blocks=b * L // 16, max_nodes=n,
                          total_nodes=b * n, max_prefix_len=L, softmax_scale=0.0, out_dtype=0)
        assert tv.attention_workspace_size(p) <= lib_scratch_bytes()
        assert tv.attention_plan(p, sms=251)["workspace_bytes"] <= lib_scratch_bytes()
        big = tv.attention_plan(p, sms=260)
        assert (big["workspace_bytes"] > lib_scratch_bytes()) == (big["ctas"] > 251)
