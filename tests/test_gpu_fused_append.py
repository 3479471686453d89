"""pkv_paged_decode_attention_append: the KV append fused into decode attention.

The call must leave the caches, the output and the status word exactly as
pkv_kv_append followed by pkv_paged_decode_attention leave them, on the fast
path (the attention kernel writes each new token into its last block just
before loading that block) and on the fallbacks (fp32, unaligned new rows),
with malformed rows included; and its output must match the oracle's append
followed by the oracle's attention.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from paged_kv_decode_table_gb300 import workloads as W
from tests.gpu_helpers import TOL, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()


def _clone(inp):
    return {k: (v.clone() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _separate(inp, bt, sl):
    st = pkv.new_status()
    pkv.kv_append(inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], bt, sl, status=st)
    out = pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], bt, sl, status=st)
    return out, st


def _fused(inp, bt, sl):
    st = pkv.new_status()
    out = pkv.paged_decode_attention_append(inp["q"], inp["k_new"], inp["v_new"], inp["k_cache"],
                                            inp["v_cache"], bt, sl, status=st)
    return out, st


def _same(a, b, oa, ob, sa, sb):
    torch.cuda.synchronize()
    assert pkv.check_status(sa) == pkv.check_status(sb)
    for key in ("k_cache", "v_cache"):
        assert torch.equal(a[key].view(torch.int16) if a[key].dtype == torch.bfloat16 else a[key],
                           b[key].view(torch.int16) if b[key].dtype == torch.bfloat16 else b[key]), key
    assert torch.equal(oa.view(torch.int16) if oa.dtype == torch.bfloat16 else oa,
                       ob.view(torch.int16) if ob.dtype == torch.bfloat16 else ob)


CASES = [(2, {}, "b64-32q8kv"), (2, dict(batch=9, len_lo=1, len_hi=900), "short-and-one-token"),
         (4, dict(batch=37), "b37-frag"), (3, dict(batch=3, len_lo=20000, len_hi=40000), "long-64q8kv"),
         (1, {}, "tiny-f32-fallback")]


@pytest.mark.parametrize("num,over,label", CASES, ids=[c[2] for c in CASES])
def test_fused_equals_append_then_attention(num, over, label):
    w = W.workload(num, **over)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    K0, V0 = host(inp["k_cache"]), host(inp["v_cache"])
    a, b = _clone(inp), _clone(inp)
    oa, sa = _separate(a, inp["block_tables"], inp["seq_lens"])
    ob, sb = _fused(b, inp["block_tables"], inp["seq_lens"])
    _same(a, b, oa, ob, sa, sb)
    assert pkv.check_status(sb) == 0
    # and against the oracle: its append, then its attention on the appended cache
    assert oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), K0, V0, host(inp["block_tables"]),
                            host(inp["seq_lens"]), w.block_size) == 0
    np.testing.assert_array_equal(host(b["k_cache"]), K0)
    np.testing.assert_array_equal(host(b["v_cache"]), V0)
    B, Hq, D = ob.shape
    rows = np.sort(np.random.default_rng(7).choice(B * Hq, size=min(B * Hq, 96), replace=False))
    ref, _, _ = oracle.paged_attention(host(inp["q"]), K0, V0, host(inp["block_tables"]),
                                       host(inp["seq_lens"]), rows=rows)
    got = ob.float().cpu().numpy().reshape(B * Hq, D)[rows]
    atol, rtol = TOL[w.dtype]
    assert np.all(np.abs(got - ref.reshape(-1, D)) <= atol + rtol * np.abs(ref.reshape(-1, D)))


def test_fused_with_unaligned_new_rows_falls_back():
    w = W.workload(2, batch=6, len_lo=20, len_hi=400)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    B, Hkv, D = inp["k_new"].shape
    for key in ("k_new", "v_new"):  # the same values, 2 bytes past a 16-byte boundary
        buf = torch.empty(B * Hkv * D + 1, dtype=inp[key].dtype, device="cuda")
        view = buf[1:].view(B, Hkv, D)
        view.copy_(inp[key])
        inp[key] = view
    a, b = _clone(inp), _clone(inp)
    a["k_new"], a["v_new"], b["k_new"], b["v_new"] = inp["k_new"], inp["v_new"], inp["k_new"], inp["v_new"]
    oa, sa = _separate(a, inp["block_tables"], inp["seq_lens"])
    ob, sb = _fused(b, inp["block_tables"], inp["seq_lens"])
    _same(a, b, oa, ob, sa, sb)
    assert pkv.check_status(sb) == 0


def test_fused_bad_rows_and_shared_prefix():
    """Malformed rows are skipped and reported as the two calls do; sequences
    sharing full prefix blocks (their last blocks private) are unaffected."""
    w = W.workload(2, batch=12, len_lo=200, len_hi=900)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    BS = w.block_size
    sl = inp["seq_lens"].clone()
    bt = inp["block_tables"].clone()
    sl[1] = 0                                        # nothing to append, nothing to attend
    sl[2] = w.max_blocks * BS + 1                    # beyond the table
    bt[3, (int(sl[3]) - 1) // BS] = inp["num_blocks"] + 5   # bad last block
    bt[4, 0] = -1                                    # bad first block, valid last block
    shared = min((int(sl[5]) - 1) // BS, (int(sl[6]) - 1) // BS)
    bt[6, :shared] = bt[5, :shared]                  # 6 reads 5's full prefix blocks
    a, b = _clone(inp), _clone(inp)
    oa, sa = _separate(a, bt, sl)
    ob, sb = _fused(b, bt, sl)
    _same(a, b, oa, ob, sa, sb)
    assert pkv.check_status(sb) == 4
    K0, V0 = host(inp["k_cache"]), host(inp["v_cache"])
    assert oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), K0, V0, host(bt), host(sl), BS) == 4
    np.testing.assert_array_equal(host(b["k_cache"]), K0)
    np.testing.assert_array_equal(host(b["v_cache"]), V0)
    ok = [r for r in range(w.batch) if r not in (1, 2, 3, 4)]
    Hq, D = inp["q"].shape[1], inp["q"].shape[2]
    rows = np.array([r * Hq + h for r in ok for h in (0, Hq - 1)])
    ref, _, _ = oracle.paged_attention(host(inp["q"]), K0, V0, host(bt), host(sl), rows=rows)
    got = ob.float().cpu().numpy().reshape(-1, D)[rows]
    atol, rtol = TOL["bf16"]
    assert np.all(np.abs(got - ref.reshape(-1, D)) <= atol + rtol * np.abs(ref.reshape(-1, D)))
