"""A bounded wait that runs out reports PKV_ERR_TIMEOUT and leaves the GPU usable.

Failure detection by a bounded wait: every mbarrier wait in the attention
kernel gives up after a poll budget and records PKV_ERR_TIMEOUT in the status
word instead of hanging.  The test hook pkv_test_set_wait_limit makes one CTA's
loader issue no copy at all (so nothing is in flight when its consumers give
up) and shortens the budget to a few polls; the call must then report
PKV_ERR_TIMEOUT, and the next call with the hook reset, on the same stream,
must match the float64 oracle.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import compare_attention
from paged_kv_decode_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()
    yield
    pkv.test_set_wait_limit()


def test_wait_runs_out_then_next_call_is_correct():
    w = W.workload(2, batch=16, len_lo=300, len_hi=2500)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    st = pkv.new_status()
    try:
        pkv.test_set_wait_limit(64, 0)      # CTA 0 (it always has blocks here) stays silent
        pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                                   inp["seq_lens"], status=st)
        torch.cuda.synchronize()
        assert pkv.check_status(st) == 5, pkv.status_string(pkv.check_status(st))
    finally:
        pkv.test_set_wait_limit()
    st2 = pkv.new_status()
    out = pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                                     inp["seq_lens"], status=st2)
    torch.cuda.synchronize()
    assert pkv.check_status(st2) == 0
    B, Hq, _ = out.shape
    rows = np.sort(np.random.default_rng(1).choice(B * Hq, size=96, replace=False))
    compare_attention(out, inp, "bf16", rows=rows)


def test_hook_rejects_bad_cta_index():
    with pytest.raises(pkv.PkvError):
        pkv.test_set_wait_limit(64, -2)
