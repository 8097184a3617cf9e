"""The device-timeout path on the GPU, without a fault: a kernel waits on an
mbarrier that nothing arrives at, through the library's bounded wait, and
must report TV_ERR_DEVICE_TIMEOUT after about the requested limit; the
context must stay usable (a tree attention call right after it is exact)."""
import numpy as np
import pytest

import speculative_decoding_tree_attention_gb300 as tv
import oracle
from speculative_decoding_tree_attention_gb300 import workloads as wl
from tv_testlib import assert_attention_close, ensure_built, run_attention

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [5.0, 50.0])
def test_wait_runs_out_and_reports(limit_ms):
    ensure_built()
    status, waited = tv.selftest_wait_timeout(limit_ms)
    assert status == tv.TV_ERR_DEVICE_TIMEOUT
    assert limit_ms * 1e6 <= waited < limit_ms * 1e6 + 200e6
    # the context is still usable
    case = wl.make_case(wl.config(1), parts=("attn",))
    gpu, st = run_attention(case)
    assert np.all(st == 0)
    assert_attention_close(gpu, oracle.tree_attention(case), "after a timeout")
