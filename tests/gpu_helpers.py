"""Shared helpers for the GPU parity tests: host copies and oracle comparisons."""
import json
import os

import numpy as np
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv

# bf16 attention: spec bar max-abs 2e-2 / rel 2e-2; fp32: 1e-5.
TOL = {"bf16": (2e-2, 2e-2), "f32": (1e-5, 1e-5)}
# Sampled tokens must match the oracle exactly unless u lies within 1e-6 of a CDF
# edge, or the top-p cut lies within 1e-6 of p (then the row is exempt and counted).
EXEMPT = 1e-6


def host(t: torch.Tensor) -> np.ndarray:
    """Host copy for the oracle: bf16 as uint16 bit patterns, others as-is."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def run_attention(inp, status=None):
    return pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                                      inp["seq_lens"], status=status)


def compare_attention(out_gpu, inp, dtype: str, rows=None):
    """Returns (max_abs_err, n_checked); asserts the tolerance element by element."""
    q, K, V = host(inp["q"]), host(inp["k_cache"]), host(inp["v_cache"])
    bt, sl = host(inp["block_tables"]), host(inp["seq_lens"])
    ref, st, werr = oracle.paged_attention(q, K, V, bt, sl, rows=rows)
    assert werr < 1e-9
    got = out_gpu.float().cpu().numpy()
    B, Hq, D = got.shape
    got = got.reshape(B * Hq, D)
    ref = ref.reshape(-1, D)
    if rows is not None:
        got = got[np.asarray(rows)]
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{int(bad.sum())} elements out of tolerance; max err {err.max():.3e}"
    return float(err.max()), got.shape[0]


def sampler_args(s):
    return (s["logits"], s["temperature"], s["top_k"], s["top_p"], s["seeds"], s["offsets"])


def compare_tokens(tokens_gpu, s):
    """Asserts token parity with exemptions; returns dict of counts."""
    res = oracle.sample_batch(host(s["logits"]), host(s["temperature"]), host(s["top_k"]),
                              host(s["top_p"]), host(s["seeds"]).view(np.uint64),
                              host(s["offsets"]).view(np.uint64))
    got = tokens_gpu.cpu().numpy()
    mism = got != res["tokens"]
    draw_ex = res["draw_margin"] < EXEMPT
    cut_ex = res["cut_margin"] < EXEMPT
    exempt = draw_ex | cut_ex
    bad = mism & ~exempt
    assert not bad.any(), (f"{int(bad.sum())} token mismatches outside the exemption: rows "
                           f"{np.nonzero(bad)[0][:10].tolist()} gpu {got[bad][:10].tolist()} "
                           f"oracle {res['tokens'][bad][:10].tolist()}")
    # an exempt mismatch must still be a token the oracle could have chosen: finite logit
    logits = host(s["logits"])
    for r in np.nonzero(mism & exempt)[0]:
        assert 0 <= got[r] < logits.shape[1] and np.isfinite(logits[r, got[r]])
    return dict(rows=int(got.shape[0]), mismatches=int(mism.sum()), exempt_draw=int(draw_ex.sum()),
                exempt_cut=int(cut_ex.sum()), exempt_mismatch=int((mism & exempt).sum()),
                status=res["status"])


def record(name: str, counts: dict) -> None:
    """Append one JSON line of parity counts to the file named by the
    PKV_PARITY_RECORD environment variable (no-op when it is unset)."""
    path = os.environ.get("PKV_PARITY_RECORD")
    if not path:
        return
    row = {"case": name}
    row.update({k: (v.tolist() if isinstance(v, np.ndarray) else v) for k, v in counts.items() if k != "status"})
    with open(path, "a") as f:
        f.write(json.dumps(row) + "\n")
