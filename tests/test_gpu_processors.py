"""GPU parity of the sampler variants: pkv_apply_logits_processors (constraint
masks, repetition / frequency / presence penalties) bit-exact against the
oracle's processors on the whole logits batch, and min-p in pkv_sample_tokens_ex
against the oracle's sampler (same token unless the oracle's decision was within
1e-6 of a CDF edge, a top-p cut or the min-p threshold; exemptions counted).
Inputs: seeded logits, random masks and per-row penalty lists.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import EXEMPT, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _processor_inputs(B, V, seed, with_mask=True, with_pen=True):
    rng = np.random.default_rng(seed)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    logits = torch.randn((B, V), generator=g, device="cuda") * 2.0
    words = (V + 31) // 32
    mask = None
    if with_mask:
        bits = rng.random((B, words * 32)) < 0.6
        bits[:, 0] = True
        m = np.zeros((B, words), np.uint64)
        for j in range(32):
            m |= bits[:, j::32].astype(np.uint64) << np.uint64(j)
        mask = m.astype(np.uint32)
    pen = None
    if with_pen:
        rp, tk, ct = [0], [], []
        for b in range(B):
            n = int(rng.integers(0, 200))
            t = rng.choice(V, size=n, replace=False)
            tk += t.tolist()
            ct += rng.integers(0, 6, n).tolist()
            rp.append(len(tk))
        rep = rng.uniform(0.5, 2.0, B).astype(np.float32)
        rep[::4] = 1.0
        pen = dict(row_ptr=np.array(rp, np.int32), tokens=np.array(tk, np.int32), counts=np.array(ct, np.int32),
                   rep=rep, freq=rng.uniform(0, 1, B).astype(np.float32),
                   pres=rng.uniform(-0.5, 1, B).astype(np.float32))
    return logits, mask, pen


def _gpu_process(logits, mask, pen, status=None):
    cu = lambda a, dt=None: None if a is None else torch.from_numpy(a.view(np.int32) if dt else a).cuda()
    kw = {}
    if mask is not None:
        kw["allow_mask"] = cu(mask, True)
    if pen is not None:
        kw.update(row_ptr=cu(pen["row_ptr"]), tokens=cu(pen["tokens"]), counts=cu(pen["counts"]),
                  repetition=cu(pen["rep"]), frequency=cu(pen["freq"]), presence=cu(pen["pres"]))
    pkv.apply_logits_processors(logits, status=status, **kw)


@pytest.mark.parametrize("B,V,with_mask,with_pen", [(16, 5000, True, True), (8, 128256, True, True),
                                                    (5, 999, False, True), (7, 77, True, False)])
def test_processors_bit_exact(B, V, with_mask, with_pen):
    logits, mask, pen = _processor_inputs(B, V, seed=B * 7 + V, with_mask=with_mask, with_pen=with_pen)
    ref = host(logits)
    st = pkv.new_status()
    _gpu_process(logits, mask, pen, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    p = pen or {}
    assert oracle.process_logits(ref, mask=mask, row_ptr=p.get("row_ptr"), tokens=p.get("tokens"),
                                 counts=p.get("counts"), rep=p.get("rep"), freq=p.get("freq"),
                                 pres=p.get("pres")) == oracle.OK
    got = host(logits)
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_processor_errors():
    logits, _, pen = _processor_inputs(3, 500, seed=1, with_mask=False)
    pen["tokens"][0] = 500
    pen["rep"][1] = 0.0
    st = pkv.new_status()
    _gpu_process(logits, None, pen, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 1


@pytest.mark.parametrize("B,V", [(64, 128256), (8, 32000), (32, 4099)])
def test_min_p_matches_oracle(B, V):
    rng = np.random.default_rng(B + V)
    logits, mask, _ = _processor_inputs(B, V, seed=V + 3, with_pen=False)
    _gpu_process(logits, mask, None)          # some tokens banned: min-p on a masked row
    temp = rng.choice([0.0, 0.5, 1.0, 1.5], B).astype(np.float32)
    top_k = rng.choice([0, 20, 1000], B).astype(np.int32)
    top_p = rng.choice([1.0, 0.9], B).astype(np.float32)
    min_p = rng.choice([0.0, 0.05, 0.3, 0.9, 1.0], B).astype(np.float32)
    seeds = rng.integers(-2**63, 2**63 - 1, B, dtype=np.int64)
    offs = np.zeros(B, np.int64)
    cu = lambda a: torch.from_numpy(a).cuda()
    st = pkv.new_status()
    tok = pkv.sample_tokens(logits, cu(temp), cu(top_k), cu(top_p), cu(seeds), cu(offs), status=st,
                            min_p=cu(min_p))
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    z = host(logits)
    got = tok.cpu().numpy()
    exempt = 0
    for b in range(B):
        r = oracle.sample_row(z[b], temp[b], top_k[b], top_p[b], int(seeds[b].view(np.uint64)), 0,
                              min_p=float(min_p[b]))
        assert r["status"] == 0
        if got[b] != r["token"]:
            assert min(r["draw_margin"], r["cut_margin"]) < EXEMPT, (b, got[b], r)
            exempt += 1
        assert np.isfinite(z[b, got[b]])
        if temp[b] > 0 and min_p[b] > 0:
            zmax = float(z[b][np.isfinite(z[b])].max())
            assert z[b, got[b]] >= zmax + temp[b] * np.log(min_p[b]) - 1e-5
    assert exempt <= max(1, B // 50)


def test_min_p_errors():
    B, V = 4, 300
    logits = torch.randn((B, V), device="cuda")
    cu = lambda a: torch.tensor(a).cuda()
    st = pkv.new_status()
    tok = pkv.sample_tokens(logits, cu([1.0] * B), torch.zeros(B, dtype=torch.int32, device="cuda"),
                            cu([1.0] * B), cu([1, 2, 3, 4]), cu([0] * B),
                            status=st, min_p=cu([0.5, 1.5, float("nan"), 0.0]))
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 1
    t = tok.cpu().tolist()
    assert t[1] == -1 and t[2] == -1 and t[0] >= 0 and t[3] >= 0
