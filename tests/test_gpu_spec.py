"""GPU parity of pkv_spec_verify against the float64 oracle (oracle.spec_verify_row).

Per request the number of accepted drafts, the emitted tokens and the rolled-back
length must equal the oracle's.  A request is exempt (and counted) only when the
oracle's decision was within 1e-6 of an edge: an acceptance test with
|u - p/q| < 1e-6, or a final draw within 1e-6 of a CDF edge; greedy requests are
never exempt.  Inputs: seeded target / draft logits (half the requests with a
draft close to the target, so that long accepted runs occur, half independent),
draft tokens picked among each draft row's 8 largest logits, mixed
temperatures (0 included), random 64-bit seeds.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv

pytestmark = pytest.mark.gpu
EXEMPT = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _inputs(B, gamma, V, seed, temps=(0.0, 0.7, 1.0, 1.3)):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    tgt = torch.randn((B, gamma + 1, V), generator=g, device="cuda") * 2.0
    noise = torch.randn((B, gamma, V), generator=g, device="cuda")
    close = (torch.arange(B, device="cuda") % 2 == 0).view(B, 1, 1)
    drf = torch.where(close, tgt[:, :gamma] + 0.3 * noise, 2.0 * noise)
    rng = np.random.default_rng(seed)
    top = torch.topk(drf, 8, dim=2).indices.cpu().numpy()
    pick = rng.integers(0, 8, (B, gamma))
    x = np.take_along_axis(top, pick[..., None], axis=2)[..., 0].astype(np.int32)
    temp = np.array([temps[i % len(temps)] for i in range(B)], np.float32)
    seeds = rng.integers(-2**63, 2**63 - 1, B, dtype=np.int64)
    offs = rng.integers(0, 2**40, B, dtype=np.int64)
    seq = rng.integers(gamma, 5000, B).astype(np.int32)
    return dict(target=tgt.contiguous(), draft=drf.contiguous(), x=torch.from_numpy(x).cuda(),
                seq=torch.from_numpy(seq).cuda(), temp=torch.from_numpy(temp).cuda(),
                seeds=torch.from_numpy(seeds).cuda(), offs=torch.from_numpy(offs).cuda())


def _run(inp, status=None):
    return pkv.spec_verify(inp["target"], inp["draft"], inp["x"], inp["seq"], inp["temp"], inp["seeds"],
                           inp["offs"], status=status)


def _compare(inp, tok, nacc, slo):
    zt, zd = inp["target"].cpu().numpy(), inp["draft"].cpu().numpy()
    x, seq, temp = inp["x"].cpu().numpy(), inp["seq"].cpu().numpy(), inp["temp"].cpu().numpy()
    seeds = inp["seeds"].cpu().numpy().view(np.uint64)
    offs = inp["offs"].cpu().numpy().view(np.uint64)
    tok, nacc, slo = tok.cpu().numpy(), nacc.cpu().numpy(), slo.cpu().numpy()
    exempt, accepted = 0, 0
    for b in range(zt.shape[0]):
        r = oracle.spec_verify_row(zt[b], zd[b], x[b], float(temp[b]), int(seeds[b]), int(offs[b]), int(seq[b]))
        assert r["status"] == 0
        same = r["n_acc"] == nacc[b] and (r["tokens"] == tok[b]).all() and r["seq_len_out"] == slo[b]
        if not same:
            assert temp[b] > 0, f"greedy request {b} differs"
            assert min(r["test_margin"], r["draw_margin"]) < EXEMPT, (b, r, tok[b], nacc[b])
            exempt += 1
        accepted += int(nacc[b])
    return exempt, accepted


@pytest.mark.parametrize("B,gamma,V", [(32, 4, 1000), (24, 3, 999), (8, 0, 513), (16, 6, 40000)])
def test_spec_verify_matches_oracle(B, gamma, V):
    inp = _inputs(B, gamma, V, seed=B * 100 + V)
    st = pkv.new_status()
    tok, nacc, slo = _run(inp, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    exempt, accepted = _compare(inp, tok, nacc, slo)
    assert exempt <= max(1, B // 50)
    if gamma:
        assert 0 < accepted < B * gamma   # both outcomes occur
    tok2, nacc2, slo2 = _run(inp)
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2) and torch.equal(nacc, nacc2) and torch.equal(slo, slo2)  # deterministic


def test_spec_verify_full_vocabulary():
    inp = _inputs(64, 4, 128256, seed=77)
    tok, nacc, slo = _run(inp)
    torch.cuda.synchronize()
    exempt, accepted = _compare(inp, tok, nacc, slo)
    assert exempt <= 2 and accepted > 0


def test_spec_verify_largest_vocabulary():
    # the largest vocabulary the entry point takes (2^23); three requests, so
    # only parity is checked (not that both outcomes occur)
    inp = _inputs(3, 2, 1 << 23, seed=5)
    tok, nacc, slo = _run(inp)
    torch.cuda.synchronize()
    exempt, _ = _compare(inp, tok, nacc, slo)
    assert exempt <= 1


def test_spec_verify_errors():
    B, gamma, V = 6, 2, 300
    inp = _inputs(B, gamma, V, seed=5, temps=(1.0,))
    inp["target"][1, 2, 7] = float("nan")
    inp["temp"][2] = -1.0
    inp["x"][3, 1] = V
    inp["seq"][4] = 1
    st = pkv.new_status()
    tok, nacc, slo = _run(inp, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) in (1, 6)
    t, n, s = tok.cpu().numpy(), nacc.cpu().numpy(), slo.cpu().numpy()
    seq = inp["seq"].cpu().numpy()
    for b in (1, 2, 3, 4):
        assert (t[b] == -1).all() and n[b] == 0 and s[b] == seq[b]
    for b in (0, 5):
        assert t[b, n[b]] >= 0 and s[b] == seq[b] - gamma + n[b]
