"""GPU parity of typical sampling (pkv_sample_tokens_typical) against the
oracle's oracle.sample_row_typical (the literal float64 definition): the same
token unless the oracle's decision was within 1e-6 of a CDF edge or of the
typical_p cut, or its boundary token within 1e-6 nats (in d) of its nearest
neighbour with a different logit, where rounding decides the order
(exemptions counted).
Inputs: seeded rows shaped like the sampler workloads (Gaussian logits of
several widths, peaked rows, nearly flat rows, banned tokens), random
temperatures and typical_p, plus constructed rows that take every branch:
two maxima 1e-3 apart, a cut inside a block of equal logits, uniform rows,
windows of more than 2048 logits, greedy rows, typical_p >= 1, and invalid
arguments.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import EXEMPT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _run(z, T, tp, seeds, offs):
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = pkv.new_status()
    tok = pkv.sample_tokens_typical(cu(z.astype(np.float32)), cu(T.astype(np.float32)),
                                    cu(tp.astype(np.float32)), cu(seeds.view(np.int64)), cu(offs.view(np.int64)),
                                    status=st)
    tok2 = pkv.sample_tokens_typical(cu(z.astype(np.float32)), cu(T.astype(np.float32)),
                                     cu(tp.astype(np.float32)), cu(seeds.view(np.int64)), cu(offs.view(np.int64)))
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2), "not deterministic"
    return tok.cpu().numpy(), pkv.check_status(st)


def _compare(z, T, tp, seeds, offs, max_exempt=None):
    got, st = _run(z, T, tp, seeds, offs)
    assert st == 0
    B = z.shape[0]
    exempt = 0
    for b in range(B):
        r = oracle.sample_row_typical(z[b], float(T[b]), float(tp[b]), int(seeds[b]), int(offs[b]))
        assert r["status"] == 0
        if got[b] != r["token"]:
            assert (r["draw_margin"] < EXEMPT or r["cut_margin"] < EXEMPT
                    or r["order_margin"] < EXEMPT), (b, int(got[b]), r)
            exempt += 1
        assert np.isfinite(z[b, got[b]])
    assert exempt <= (max_exempt if max_exempt is not None else max(1, B // 50))
    return exempt


@pytest.mark.parametrize("B,V,seed", [(64, 128256, 1), (32, 32000, 2), (16, 152064, 3), (40, 4099, 4), (8, 300001, 5),
                                      (2, 1 << 23, 6)])  # the largest vocabulary the entry point takes
def test_typical_matches_oracle(B, V, seed):
    rng = np.random.default_rng(seed)
    z = np.empty((B, V), np.float32)
    for b in range(B):
        kind = b % 4
        if kind == 0:
            z[b] = rng.standard_normal(V) * 2.0
        elif kind == 1:
            z[b] = rng.standard_normal(V)
            z[b, rng.integers(V)] += 12.0                     # peaked
        elif kind == 2:
            z[b] = rng.standard_normal(V) * 0.1               # nearly flat
        else:
            z[b] = rng.standard_normal(V) * 1.5
            z[b, rng.random(V) < 0.3] = -np.inf               # banned tokens
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[::7] = 0.0
    tp = rng.choice([0.2, 0.5, 0.9, 0.95, 1.0], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    e = _compare(z, T, tp, seeds, offs)
    print(f"typical B={B} V={V}: exempt mismatches {e}")


def test_constructed_rows():
    V = 1000
    rows, T, tp = [], [], []

    def add(z, t, p):
        rows.append(np.asarray(z, np.float32))
        T.append(t)
        tp.append(p)
    # 998 equal logits far below two maxima 1e-3 apart (the cut falls on them
    # at 0.97 / 0.99); inside the block of equal logits the cut is the r-th
    # id (0.5)
    base = np.full(V, -3.0, np.float32)
    base[10] = 0.0
    base[700] = np.float32(-1e-3)
    for p in (0.5, 0.97, 0.99, 0.96):
        add(base, 1.0, p)
    for p in (0.1, 0.5, 0.77):                       # uniform rows: the first ceil(p n) ids
        add(np.full(V, 0.25, np.float32), 0.8, p)
    zb = np.full(V, -np.inf, np.float32)
    zb[[3, 400, 999]] = [1.0, 1.0, 0.5]               # three finite logits
    add(zb, 1.0, 0.6)
    add(zb, 0.0, 0.6)                                 # greedy: lowest id of the maximum
    rng = np.random.default_rng(9)
    add(rng.standard_normal(V).astype(np.float32), 1.2, 1.0)   # no truncation
    z = np.stack(rows)
    B = z.shape[0]
    Tn, tpn = np.array(T, np.float32), np.array(tp, np.float32)
    for s in range(6):
        seeds = np.arange(B, dtype=np.uint64) * 7919 + s
        offs = np.full(B, s, np.uint64)
        _compare(z, Tn, tpn, seeds, offs, max_exempt=1)
    # typical_p >= 1 is the plain draw of pkv_sample_tokens (same uniform)
    cu = lambda a: torch.from_numpy(a).cuda()
    seeds = np.arange(B, dtype=np.uint64)
    offs = np.zeros(B, np.uint64)
    a, _ = _run(z, Tn, np.ones(B, np.float32), seeds, offs)
    b = pkv.sample_tokens(cu(z), cu(Tn), torch.zeros(B, dtype=torch.int32, device="cuda"),
                          cu(np.ones(B, np.float32)), cu(seeds.view(np.int64)), cu(offs.view(np.int64)))
    assert np.array_equal(a, b.cpu().numpy())


def test_rows_past_the_window():
    """More than 2048 logits around the cut (the window path cannot hold them):
    a uniform row of 5000, and a row of two populations (T = log2(e) makes
    u = z - zmax: 130 logits at u = 0 and 2080 at u = -4.25, whose p-weighted
    mean -1.94 puts the first population at D = 1.94 and the second, whose
    2080 equal logits share one window bin, at D = 2.31; thresholds above 0.54
    cut inside the second, in id order)."""
    V = 5000
    rows, T, tp = [], [], []
    for p in (0.2001, 0.6131):
        rows.append(np.full(V, -1.5, np.float32))
        T.append(1.0)
        tp.append(p)
    z = np.full(V, -np.inf, np.float32)
    rng = np.random.default_rng(4)
    pos = rng.permutation(V)[:2210]
    z[pos[:130]] = 0.0
    z[pos[130:]] = -4.25
    for p in (0.31, 0.81, 0.999):
        rows.append(z.copy())
        T.append(1.4426950408889634)
        tp.append(p)
    zz = np.stack(rows)
    B = zz.shape[0]
    for s in range(4):
        _compare(zz, np.array(T, np.float32), np.array(tp, np.float32), np.arange(B, dtype=np.uint64) + 11 * s,
                 np.full(B, s, np.uint64), max_exempt=0)


def test_typical_errors():
    V = 300
    z = np.random.default_rng(1).standard_normal((5, V)).astype(np.float32)
    z[4, 7] = np.nan
    T = np.array([1.0, 1.0, -1.0, 0.0, 1.0], np.float32)
    tp = np.array([0.0, np.nan, 0.5, 0.0, 0.5], np.float32)
    got, st = _run(z, T, tp, np.arange(5, dtype=np.uint64), np.zeros(5, np.uint64))
    assert st in (1, 6)
    assert got[0] == -1 and got[1] == -1 and got[2] == -1 and got[4] == -1
    assert got[3] == int(np.argmax(z[3]))           # greedy ignores typical_p
