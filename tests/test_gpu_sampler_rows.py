"""GPU parity of the sampler on batches with more rows than the cluster kernel
keeps resident (B > 2 x #SM, V <= 65536): those take the one-CTA-per-row
kernel (sampler_rows.cu).  Every row is compared with the float64 oracle: the
same token unless the oracle's draw or top-p cut lies within 1e-6 of an edge
(counted, at most max(1, B // 50)).  Rows cover greedy, top-k from 1 to past the
finite count, top-p from 0.3 to 1, min-p, banned tokens, rows that are not
16-byte aligned (odd vocabularies), windows too large for the gather (blocks of
equal logits, which take the exact radix selection), the error codes, and
batches in any row order (the kernel picks the order its CTAs take the rows in).
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


def _rows():
    return 2 * torch.cuda.get_device_properties(0).multi_processor_count + 16


def _run(z, T, k, p, seeds, offs, min_p=None):
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    st = pkv.new_status()
    args = (cu(z), cu(T), cu(k), cu(p), cu(seeds.view(np.int64)), cu(offs.view(np.int64)))
    tok = pkv.sample_tokens(*args, status=st, min_p=None if min_p is None else cu(min_p))
    tok2 = pkv.sample_tokens(*args, min_p=None if min_p is None else cu(min_p))
    torch.cuda.synchronize()
    assert torch.equal(tok, tok2), "not deterministic"
    return tok.cpu().numpy(), pkv.check_status(st)


def _compare(z, T, k, p, seeds, offs, min_p=None, max_exempt=None):
    got, st = _run(z, T, k, p, seeds, offs, min_p)
    assert st == 0, pkv.status_string(st)
    B = z.shape[0]
    exempt = 0
    for b in range(B):
        r = oracle.sample_row(z[b], float(T[b]), int(k[b]), float(p[b]), int(seeds[b]), int(offs[b]),
                              min_p=0.0 if min_p is None else float(min_p[b]))
        assert r["status"] == 0
        if got[b] != r["token"]:
            assert r["draw_margin"] < EXEMPT or r["cut_margin"] < EXEMPT, (b, int(got[b]), r)
            exempt += 1
    assert exempt <= (max_exempt if max_exempt is not None else max(1, B // 50))
    return exempt


def _params(rng, B, V):
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[::9] = 0.0
    k = rng.choice([0, 0, 1, 5, 50, 1000, V - 1, V + 7], B).astype(np.int32)
    p = rng.choice([0.3, 0.8, 0.95, 1.0], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    return T, k, p, seeds, offs


@pytest.mark.parametrize("V,seed", [(32000, 1), (1001, 2), (65536, 3), (4099, 4)])
def test_rows_match_oracle(V, seed):
    rng = np.random.default_rng(seed)
    B = _rows()
    z = (rng.standard_normal((B, V)) * rng.choice([0.1, 1.0, 1.5, 3.0], (B, 1))).astype(np.float32)
    z[1::5, : V // 3] = -np.inf                                        # banned tokens
    z[2::7, rng.integers(V)] += 12.0                                   # peaked rows
    T, k, p, seeds, offs = _params(rng, B, V)
    e = _compare(z, T, k, p, seeds, offs)
    print(f"rows B={B} V={V}: exempt mismatches {e}")


def test_rows_min_p():
    rng = np.random.default_rng(7)
    B, V = _rows(), 20000
    z = (rng.standard_normal((B, V)) * 1.5).astype(np.float32)
    T, k, p, seeds, offs = _params(rng, B, V)
    mp = rng.choice([0.0, 0.05, 0.3, 0.9, 1.0], B).astype(np.float32)
    _compare(z, T, k, p, seeds, offs, min_p=mp)


def test_rows_large_windows_and_ties():
    """Blocks of equal logits larger than the gather window (the exact radix
    path), top-k boundaries inside a tie, single-logit rows, uniform rows."""
    rng = np.random.default_rng(11)
    B, V = _rows(), 6000
    z = np.empty((B, V), np.float32)
    T = np.full(B, 1.0, np.float32)
    k = np.zeros(B, np.int32)
    p = np.ones(B, np.float32)
    for b in range(B):
        kind = b % 6
        if kind == 0:                       # uniform row: every bin holds all logits
            z[b] = 0.5
            p[b] = rng.choice([0.20013, 0.50021, 0.90007])   # p * V not near an integer
        elif kind == 1:                     # two values; the cut inside the lower block of 5000
            z[b] = -1.0
            z[b, rng.permutation(V)[:1000]] = 0.0
            p[b] = 0.9
        elif kind == 2:                     # top-k boundary inside a block of ties
            z[b] = rng.standard_normal(V).astype(np.float32)
            z[b, rng.permutation(V)[:300]] = 2.5
            k[b] = 120
            p[b] = rng.choice([0.5, 1.0])
        elif kind == 3:                     # a single finite logit
            z[b] = -np.inf
            z[b, rng.integers(V)] = 3.0
            p[b] = 0.5
        elif kind == 4:                     # top-k larger than the window, top-p off
            z[b] = (rng.standard_normal(V) * 0.01).astype(np.float32)
            k[b] = 4000
        else:                               # greedy over ties: the lowest id
            z[b] = rng.integers(-3, 3, V).astype(np.float32)
            T[b] = 0.0
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    _compare(z, T, k, p, seeds, offs)


def test_rows_errors():
    rng = np.random.default_rng(5)
    B, V = _rows(), 3000
    z = rng.standard_normal((B, V)).astype(np.float32)
    T = np.ones(B, np.float32)
    k = np.zeros(B, np.int32)
    p = np.full(B, 0.9, np.float32)
    z[3, 17] = np.nan
    z[4] = -np.inf
    T[5] = -1.0
    p[6] = 0.0
    seeds = np.arange(B, dtype=np.uint64)
    offs = np.zeros(B, np.uint64)
    got, st = _run(z, T, k, p, seeds, offs)
    assert st in (1, 6)
    assert got[3] == -1 and got[4] == -1 and got[5] == -1 and got[6] == -1
    ok = [b for b in range(B) if b not in (3, 4, 5, 6)]
    ref = oracle.sample_batch(z[ok], T[ok], k[ok], p[ok], seeds[ok], offs[ok])
    mism = (got[ok] != ref["tokens"]) & (ref["draw_margin"] >= EXEMPT) & (ref["cut_margin"] >= EXEMPT)
    assert not mism.any()


@pytest.mark.parametrize("V,seed", [(32000, 31), (4099, 32)])
def test_rows_small_top_k(V, seed):
    """Rows with 0 < top_k <= 64 take the thread-maxima path (candidates from
    the threads whose maximum can be in the top k): plain and peaked rows,
    min-p, top-k 1 and 64, a top-k boundary inside a block of 60 equal logits,
    blocks of 300 equal top logits (more candidates than threads: the general
    path), few finite logits, and -0.0 / +0.0 ties."""
    rng = np.random.default_rng(seed)
    B = _rows()
    z = (rng.standard_normal((B, V)) * rng.choice([0.1, 1.0, 2.0], (B, 1))).astype(np.float32)
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    k = rng.choice([1, 2, 17, 50, 63, 64], B).astype(np.int32)
    # top_p * (number of equal masses) never an integer: no cut exactly at p
    p = rng.choice([0.50021, 0.90007, 1.0], B).astype(np.float32)
    mp = np.where(rng.random(B) < 0.3, rng.choice([0.01, 0.2, 0.7], B), 0.0).astype(np.float32)
    for b in range(B):
        kind = b % 7
        if kind == 1:
            z[b, rng.integers(V)] += 12.0
        elif kind == 2:                         # boundary inside a block of 60 equal logits
            z[b, rng.permutation(V)[:60]] = 9.0
            z[b, rng.permutation(V)[:20]] = 9.5
            k[b] = 50
        elif kind == 3:                         # 300 equal top logits
            z[b, rng.permutation(V)[:300]] = 9.0
            k[b] = rng.choice([1, 64])
        elif kind == 4:                         # 40 finite logits
            z[b] = -np.inf
            z[b, rng.permutation(V)[:40]] = rng.standard_normal(40).astype(np.float32)
            k[b] = rng.choice([5, 39])
        elif kind == 5:                         # -0.0 and +0.0 on top
            z[b] = np.minimum(z[b], -3.0)
            z[b, rng.permutation(V)[:25]] = -0.0
            z[b, rng.permutation(V)[:25]] = 0.0
            k[b] = 30
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    _compare(z, T, k, p, seeds, offs)
    _compare(z, T, k, p, seeds, offs, min_p=mp)


@pytest.mark.parametrize("mix", ["mixed", "top_p_only", "heavy_tail"])
def test_rows_order_independent(mix):
    """The rows kernel hands its CTAs the rows heaviest first (top-p alone, then
    large top-k or no truncation, then greedy, small top-k and invalid rows),
    or in their natural order when every row is in one class: the token of a
    row does not depend on where it sits in the batch, so permuting the rows
    permutes the tokens.  A mixed batch, a batch of top-p rows only, and a
    batch whose only heavy rows are its last ones."""
    rng = np.random.default_rng({"mixed": 51, "top_p_only": 52, "heavy_tail": 53}[mix])
    B, V = _rows(), 6000
    z = (rng.standard_normal((B, V)) * rng.choice([0.5, 1.0, 2.0], (B, 1))).astype(np.float32)
    T, k, p, seeds, offs = _params(rng, B, V)
    if mix == "top_p_only":
        T[:] = rng.uniform(0.5, 1.5, B).astype(np.float32)
        k[:] = 0
        p[:] = 0.90007
    elif mix == "heavy_tail":
        T[:] = 0.0
        T[-20:] = 1.0
        k[-20:] = 0
        p[-20:] = 0.80007
    got, st = _run(z, T, k, p, seeds, offs)
    assert st == 0
    perm = rng.permutation(B)
    got_p, st_p = _run(z[perm], T[perm], k[perm], p[perm], seeds[perm], offs[perm])
    assert st_p == 0
    assert np.array_equal(got_p, got[perm])
    for b in list(range(0, B, 37)) + list(range(B - 20, B)):
        r = oracle.sample_row(z[b], float(T[b]), int(k[b]), float(p[b]), int(seeds[b]), int(offs[b]))
        if got[b] != r["token"]:
            assert r["draw_margin"] < EXEMPT or r["cut_margin"] < EXEMPT, (b, int(got[b]), r)


def test_rows_logits_on_bin_edges():
    """Logits on a grid of 1/256 over a range of 8: with 2048 bins over the
    row's range every logit lies exactly on a bin edge, where the passes that
    test a logit's bin by comparing it with the bin's lowest logit must agree
    with the bin itself; top-p, top-k above 64, min-p and no truncation."""
    rng = np.random.default_rng(61)
    B, V = _rows(), 4099
    grid = -np.arange(0, 2049, dtype=np.float64) / 256.0 + 3.0
    z = grid[rng.integers(0, 2049, (B, V))].astype(np.float32)
    z[:, 0] = 3.0       # the maximum and the minimum fix the range at 8
    z[:, 1] = 3.0 - 8.0
    T = rng.choice([0.25, 0.5, 1.0, 2.0], B).astype(np.float32)
    k = rng.choice([0, 0, 100, 1000], B).astype(np.int32)
    p = rng.choice([0.30011, 0.70013, 0.95003, 1.0], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    mp = np.where(rng.random(B) < 0.3, 0.01, 0.0).astype(np.float32)
    _compare(z, T, k, p, seeds, offs)
    _compare(z, T, k, p, seeds, offs, min_p=mp)
