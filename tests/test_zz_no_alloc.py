"""The allocation-free attention entry point agrees with the workspace one.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate device
memory when attention runs (all free HBM already handed to the KV pool, no
tolerance for an allocation's implicit synchronisation, or a plain C host with
no device allocator): its split-KV scratch is a fixed array inside the library.
This test drives it through the C ABI twice in a row, with different batches so
that the second call finds the first call's leftovers in the shared scratch, and
compares each result with pkv_paged_decode_attention on the same inputs: both
run the same kernels with the same split, so the outputs must be identical bit
for bit.  One case is also checked against the float64 oracle on sampled rows,
within the bf16 attention tolerance of the other parity tests.  It also checks
that a request needing more scratch than the array holds is refused without a
launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import compare_attention
from paged_kv_decode_table_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 2e-2  # bf16 attention tolerance used by the parity tests


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    L = pkv.load_library()
    P = ctypes.c_void_p
    i32, f32 = ctypes.c_int, ctypes.c_float
    L.pkv_paged_decode_attention_noalloc.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f32,
                                                     i32, P, P]
    L.pkv_paged_decode_attention_noalloc.restype = i32
    return L


def _noalloc(L, inp, out, status):
    q, k, v = inp["q"], inp["k_cache"], inp["v_cache"]
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k.shape
    bt, sl = inp["block_tables"], inp["seq_lens"]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return L.pkv_paged_decode_attention_noalloc(
        p(out), p(q), p(k), p(v), p(bt), bt.shape[1], p(sl), B, Hq, Hkv, D, BS, NB, 0.0,
        1 if q.dtype == torch.bfloat16 else 0, p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(lib):
    cases = [W.workload(2, batch=12, len_lo=200, len_hi=3000),   # sequences split across CTAs
             W.workload(3, batch=3, len_lo=2000, len_hi=9000)]   # other shape, G = 8
    for w in cases:
        inp = W.make_decode_inputs(w, "cuda", with_logits=False)
        ref = pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                                         inp["seq_lens"])
        out = torch.full_like(inp["q"], float("nan"))
        status = pkv.new_status()
        code = _noalloc(lib, inp, out, status)
        torch.cuda.synchronize()
        assert code == 0, pkv.status_string(code)
        assert pkv.check_status(status) == 0
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out, ref)
        err = (out.float() - ref.float()).abs()
        assert bool((err <= ATOL + RTOL * ref.float().abs()).all()), float(err.max())
    # the second case against the float64 oracle, 64 sampled (sequence, head) rows
    B, Hq, _ = out.shape
    rows = np.random.default_rng(0).choice(B * Hq, size=min(64, B * Hq), replace=False)
    compare_attention(out, inp, "bf16", rows=np.sort(rows))


def test_noalloc_refuses_requests_beyond_its_scratch(lib):
    w = W.workload(2, batch=4, len_lo=20, len_hi=60)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    # pretend to be a batch far larger than the scratch can hold: B * Hq * D partials
    big_B, big_Hq = 4096, 128
    assert pkv.decode_workspace_bytes(big_B, big_Hq, 128) > (16 << 20)
    q = torch.zeros(big_B, big_Hq, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    bt = torch.zeros(big_B, inp["block_tables"].shape[1], dtype=torch.int32, device="cuda")
    sl = torch.zeros(big_B, dtype=torch.int32, device="cuda")
    big = dict(q=q, k_cache=inp["k_cache"], v_cache=inp["v_cache"], block_tables=bt, seq_lens=sl)
    # Hkv of the pool is 8 and 128 % 8 == 0, so only the scratch size can refuse it
    code = _noalloc(lib, big, out, pkv.new_status())
    assert code == 2  # PKV_ERR_UNSUPPORTED, nothing launched
