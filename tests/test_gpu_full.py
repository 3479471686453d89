"""GPU parity at the full workload sizes, through the same calls the benchmark times.

Attention: every query head of the longest and the shortest sequence plus a
seeded sample of (sequence, head) rows is recomputed by the float64 oracle.
Sampler: every row is recomputed by the oracle; a token may differ only where
the oracle's draw or top-p cut lies within 1e-6 of an edge, and at most
max(1, rows // 50) rows may.  KV append: the whole pools are compared bit for
bit.  With PKV_PARITY_RECORD set, the per-workload counts (rows, mismatches,
exempt draws and cuts) are appended to that file as JSON lines.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from paged_kv_decode_table_gb300 import workloads as W
from tests.gpu_helpers import compare_attention, compare_tokens, host, record, run_attention, sampler_args

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    oracle.build()


def _sample_rows(w, seq_lens, n_random, seed):
    sl = seq_lens.cpu().numpy()
    Hq = w.n_q_heads
    rng = np.random.default_rng(seed)
    rows = set()
    for b in (int(np.argmax(sl)), int(np.argmin(sl))):
        rows.update(range(b * Hq, (b + 1) * Hq))
    rows.update(rng.choice(w.batch * Hq, size=min(n_random, w.batch * Hq), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("num,n_random", [(1, 8), (2, 256), (3, 96), (4, 512)])
def test_full_size_decode_step(num, n_random):
    w = W.workload(num)
    inp = W.make_decode_inputs(w, "cuda")
    Kh, Vh = host(inp["k_cache"]), host(inp["v_cache"])
    st = pkv.new_status()
    # the decode step as the benchmark runs it: append, attention, sampler
    pkv.kv_append(inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                  inp["seq_lens"], status=st)
    out = run_attention(inp, st)
    tok = pkv.sample_tokens(*sampler_args(inp), status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    # append: whole pools bit for bit
    oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), Kh, Vh, host(inp["block_tables"]),
                     host(inp["seq_lens"]), w.block_size)
    np.testing.assert_array_equal(host(inp["k_cache"]), Kh)
    np.testing.assert_array_equal(host(inp["v_cache"]), Vh)
    del Kh, Vh
    # attention on sampled rows
    rows = _sample_rows(w, inp["seq_lens"], n_random, seed=num)
    err, n = compare_attention(out, inp, "f32" if inp["q"].dtype == torch.float32 else "bf16", rows=rows)
    print(f"workload {num}: attention max |err| {err:.3e} over {n} rows")
    # sampler, every row
    c = compare_tokens(tok, inp)
    print(f"workload {num}: sampler {c}")
    assert c["exempt_mismatch"] <= max(1, c["rows"] // 50)
    record(f"workload {num} ({w.name}): sampler", c)
    record(f"workload {num} ({w.name}): attention", {"rows_checked": n, "max_abs_err": err})
    if num == 3:
        # T = 1e-3 is greedy-equivalent: the token is the argmax of each row
        am = torch.argmax(inp["logits"], dim=1).to(torch.int32)
        assert torch.equal(tok, am)


def test_full_size_sampler_stress():
    w = W.workload(5)
    s = W.make_sampler_inputs(w, "cuda")
    st = pkv.new_status()
    tok = pkv.sample_tokens(*sampler_args(s), status=st)
    tok2 = pkv.sample_tokens(*sampler_args(s))
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    assert torch.equal(tok, tok2)
    c = compare_tokens(tok, s)
    print(f"sampler stress: {c}")
    assert c["exempt_mismatch"] <= max(1, c["rows"] // 50)
    record(f"workload 5 ({w.name}): sampler", c)
