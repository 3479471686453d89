"""Pins of the typical-sampling oracle (oracle.sample_row_typical), CPU.

"LLM inference serving tutorial" section 3.1 (other samplers) defines typical
sampling: H(p) = -sum p ln p, d_i = |-ln p_i - H|, keep the smallest prefix in
ascending d whose cumulative probability reaches typical_p, renormalise.  Pinned
to the page's worked example ([D01], tests/golden/typical_sampling_d01.txt),
closed forms (uniform rows: H = ln n, every d = 0, so the first ceil(tau n) ids
are kept), the interval property of the kept set, shift invariance, the
typical_p >= 1 and T = 0 reductions to the pinned sampler, the definition
written out independently with numpy (small rows, and 40 rows of 128256
logits), a constructed row whose kept set changes if the centre is rounded,
and a chi-square test of the draws.
"""
import math

import numpy as np
import pytest

import oracle


def _support(r):
    return set(np.nonzero(r["probs"])[0].tolist())


def _examples(path):
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, probs, tp, exp = line.split()
        yield name, [float(x) for x in probs.split(",")], float(tp), {int(x) for x in exp.split(",")}


def test_page_example(golden_dir):
    seen = 0
    for name, probs, tp, expected in _examples(f"{golden_dir}/typical_sampling_d01.txt"):
        z = np.log(np.array(probs)).astype(np.float32)
        r = oracle.sample_row_typical(z, 1.0, tp, 7, 0, want_probs=True)
        assert r["status"] == oracle.OK, name
        assert _support(r) == expected, (name, _support(r))
        seen += 1
    assert seen == 4
    # the example's point: the most probable token is dropped, unlike top-p
    z = np.log(np.array([0.02, 0.35, 0.33, 0.30])).astype(np.float32)
    r = oracle.sample_row_typical(z, 1.0, 0.62, 7, 0, want_probs=True)
    assert 1 not in _support(r)
    top = oracle.sample_row(z, 1.0, 0, 0.62, 7, 0, want_probs=True)
    assert 1 in set(np.nonzero(top["probs"])[0].tolist())


@pytest.mark.parametrize("n,tp", [(1, 0.5), (5, 0.5), (8, 0.3), (13, 0.999), (64, 0.2), (4, 0.5), (8, 0.25)])
def test_uniform_row_closed_form(n, tp):
    z = np.full(n, 0.75, np.float32)
    r = oracle.sample_row_typical(z, 0.9, tp, 3, 1, want_probs=True)
    assert r["status"] == oracle.OK
    assert abs(r["entropy"] - math.log(n)) < 1e-12
    m = math.ceil(np.float32(tp) * n - 1e-12)
    assert _support(r) == set(range(m))
    np.testing.assert_allclose(r["probs"][:m], 1.0 / m, rtol=1e-12)
    # top-p keeps the same first m ids of a uniform row, so the pinned
    # sampler's draw (token-id order, same uniform) must agree
    for seed in range(12):
        a = oracle.sample_row_typical(z, 0.9, tp, seed, 5)
        b = oracle.sample_row(z, 0.9, 0, tp, seed, 5)
        assert a["token"] == b["token"]


def _u(z, T):
    return (z.astype(np.float64) - z.max()) / T * math.log2(math.e)


@pytest.mark.parametrize("seed", range(6))
def test_kept_set_is_an_interval_around_the_mean(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(50, 3000))
    z = (rng.standard_normal(V) * rng.uniform(0.3, 3)).astype(np.float32)
    T, tp = float(np.float32(rng.uniform(0.5, 1.5))), float(rng.uniform(0.2, 0.95))
    r = oracle.sample_row_typical(z, T, tp, seed, 0, want_probs=True)
    assert r["status"] == oracle.OK
    kept = r["probs"] > 0
    p = np.exp((z.astype(np.float64) - z.max()) / T)
    p /= p.sum()
    u = _u(z, T)
    ubar = float((p * u).sum())
    dist = np.abs(u - ubar)
    # every dropped token is at least as far from the mean as every kept one
    assert dist[~kept].min() >= dist[kept].max() - 1e-9
    # the kept mass reaches typical_p, and dropping one of the farthest kept
    # tokens would not
    assert p[kept].sum() >= np.float32(tp) - 1e-12
    band = np.nonzero(kept & (dist >= dist[kept].max() - 1e-9))[0]
    assert any(p[kept].sum() - p[j] < np.float32(tp) + 1e-12 for j in band)
    # the entropy the oracle reports is the page's H
    assert abs(r["entropy"] - float(-(p[p > 0] * np.log(p[p > 0])).sum())) < 1e-9


@pytest.mark.parametrize("seed", range(4))
def test_shift_invariance(seed):
    rng = np.random.default_rng(100 + seed)
    z = (rng.integers(-256, 256, 500) / 64.0).astype(np.float32)   # exact under the shifts below
    a = oracle.sample_row_typical(z, 0.8, 0.7, 11, 2, want_probs=True)
    for c in (-3.0, 5.0, 32.0):
        b = oracle.sample_row_typical((z + np.float32(c)).astype(np.float32), 0.8, 0.7, 11, 2, want_probs=True)
        assert _support(b) == _support(a) and b["token"] == a["token"]


def test_reductions_to_the_pinned_sampler():
    rng = np.random.default_rng(5)
    z = rng.standard_normal(300).astype(np.float32)
    for seed in range(5):
        a = oracle.sample_row_typical(z, 0.9, 1.0, seed, 3)
        b = oracle.sample_row(z, 0.9, 0, 1.0, seed, 3)
        assert a["token"] == b["token"]
        g = oracle.sample_row_typical(z, 0.0, 0.5, seed, 3)
        assert g["token"] == int(np.argmax(z))


def _literal_kept(z, T, tp):
    """The section 3.1 definition written out with numpy in float64: p, H,
    d = |-ln p - H|, ascending d (equal d: larger logit, then smaller id),
    the smallest prefix reaching typical_p.  Returns (kept ids, gap in d at
    the boundary to the nearest neighbours with a different logit)."""
    fin = np.isfinite(z)
    ids = np.nonzero(fin)[0]
    a = (z[ids].astype(np.float64) - z[ids].max()) / T
    lnp = a - math.log(np.exp(a).sum())
    p = np.exp(lnp)
    H = float(-(p * lnp).sum())
    d = np.abs(-lnp - H)
    order = np.lexsort((ids, -z[ids].astype(np.float64), d))
    cum = np.cumsum(p[order])
    m = int(np.searchsorted(cum, np.float32(tp), side="left")) + 1
    m = min(m, ids.size)
    c = m - 1
    zc, dc, gap = z[ids[order[c]]], d[order[c]], np.inf
    for j in range(c - 1, -1, -1):
        if z[ids[order[j]]] != zc:
            gap = min(gap, dc - d[order[j]])
            break
    for j in range(c + 1, ids.size):
        if z[ids[order[j]]] != zc:
            gap = min(gap, d[order[j]] - dc)
            break
    return set(ids[order[:m]].tolist()), gap


def test_literal_definition_on_small_rows():
    """Rows of 4..8 tokens, every threshold: the oracle's kept set is the
    definition's, written out independently above."""
    checked = 0
    for seed in range(60):
        rng = np.random.default_rng(200 + seed)
        V = int(rng.integers(4, 9))
        z = (rng.standard_normal(V) * 1.5).astype(np.float32)
        T = float(np.float32(rng.uniform(0.5, 1.5)))
        for tp in (0.1, 0.3, 0.5, 0.7, 0.9):
            keep, gap = _literal_kept(z, T, tp)
            if gap < 1e-12:
                continue
            r = oracle.sample_row_typical(z, T, tp, 1, 0, want_probs=True)
            assert _support(r) == keep, (seed, tp)
            checked += 1
    assert checked >= 250


@pytest.mark.parametrize("seed", range(40))
def test_literal_definition_on_vocabulary_rows(seed):
    """Rows of 128256 logits ~ N(0, 1) or N(0, 2^2), T in [0.5, 1.5],
    typical_p in {0.2, 0.5, 0.9, 0.95}: the kept set and the boundary gap are
    the definition's; the token is the draw over that set in id order."""
    rng = np.random.default_rng(7000 + seed)
    V = 128256
    z = (rng.standard_normal(V) * (1.0 if seed % 2 else 2.0)).astype(np.float32)
    T = float(np.float32(rng.uniform(0.5, 1.5)))
    tp = float(np.float32([0.2, 0.5, 0.9, 0.95][seed % 4]))
    keep, gap = _literal_kept(z, T, tp)
    r = oracle.sample_row_typical(z, T, tp, seed, 3, want_probs=True)
    assert r["status"] == oracle.OK
    if gap > 1e-12:
        assert _support(r) == keep
        assert abs(r["order_margin"] - gap) <= 1e-12
    k = np.array(sorted(_support(r)))
    pk = np.exp((z[k].astype(np.float64) - z.max()) / T)
    cdf = np.cumsum(pk / pk.sum())
    u = oracle.uniform(seed, 3)
    assert r["token"] == int(k[min(np.searchsorted(cdf, u, side="right"), k.size - 1)])


def test_centre_is_not_rounded():
    """A row whose p-weighted mean sits 0.45 of a 2^-8 step (log2 units) above
    a multiple of 2^-8: 1024 logits at 0 and 3070 at -c (T = 1) put the mean
    of a = z - z_max at abar = -c w / (1024 + w), w = 3070 e^-c; two probes sit
    at abar + 2e-4 and abar - 7e-4.  Every other token is far from abar, so in
    the definition's order the first probe comes first (d = 2e-4 against
    7e-4, each moved by about 1e-7 by the probes' own weight), and a
    typical_p below its probability keeps it alone.  A centre rounded to the
    2^-8 grid (down by 0.45 * 2^-8 * ln 2 = 1.2e-3 nats) would put the second
    probe first instead."""
    c = float(np.float32(0.8069599866867065))
    w = 3070 * math.exp(-c)
    abar = -c * w / (1024 + w)
    frac = (abar / math.log(2) * 256) % 1.0
    assert 0.40 < frac < 0.50                       # the rounding goes down by ~0.45 step
    zi, zj = np.float32(abar + 2e-4), np.float32(abar - 7e-4)
    z = np.concatenate([np.zeros(1024, np.float32), np.full(3070, -c, np.float32), [zi, zj]]).astype(np.float32)
    perm = np.random.default_rng(0).permutation(z.size)
    zz = z[perm]
    i_id, j_id = int(np.nonzero(perm == 4094)[0][0]), int(np.nonzero(perm == 4095)[0][0])
    # on the grid the second probe would be nearer the centre
    grid = math.floor(abar / math.log(2) * 256) / 256 * math.log(2)
    assert abs(float(zj) - grid) < abs(float(zi) - grid)
    for seed in range(4):
        r = oracle.sample_row_typical(zz, 1.0, 1e-4, seed, 0, want_probs=True)
        assert r["status"] == oracle.OK
        assert _support(r) == {i_id} and r["token"] == i_id
        assert abs(r["order_margin"] - 5e-4) < 1e-5
    # a threshold above the first probe's probability takes the second one next
    r = oracle.sample_row_typical(zz, 1.0, 5e-4, 0, 0, want_probs=True)
    assert _support(r) == {i_id, j_id}


def test_draws_follow_the_kept_distribution():
    rng = np.random.default_rng(9)
    z = (rng.standard_normal(40) * 1.2).astype(np.float32)
    r = oracle.sample_row_typical(z, 1.0, 0.6, 0, 0, want_probs=True)
    probs = r["probs"]
    n = 4000
    counts = np.zeros(40)
    for s in range(n):
        counts[oracle.sample_row_typical(z, 1.0, 0.6, s, 0)["token"]] += 1
    k = probs > 0
    assert counts[~k].sum() == 0
    chi2 = float((((counts[k] - n * probs[k]) ** 2) / (n * probs[k])).sum())
    dof = int(k.sum()) - 1
    assert chi2 < dof + 6 * math.sqrt(2 * dof) + 10


def test_errors():
    z = np.zeros(10, np.float32)
    assert oracle.sample_row_typical(z, 1.0, 0.0, 0, 0)["status"] == oracle.INVALID_ARG
    assert oracle.sample_row_typical(z, 1.0, float("nan"), 0, 0)["status"] == oracle.INVALID_ARG
    assert oracle.sample_row_typical(z, -1.0, 0.5, 0, 0)["status"] == oracle.INVALID_ARG
    bad = z.copy()
    bad[3] = np.nan
    assert oracle.sample_row_typical(bad, 1.0, 0.5, 0, 0)["status"] == oracle.NONFINITE
    assert oracle.sample_row_typical(np.full(4, -np.inf, np.float32), 1.0, 0.5, 0, 0)["status"] == oracle.NONFINITE
    assert oracle.sample_row_typical(z, 0.0, 0.0, 0, 0)["status"] == oracle.OK   # greedy ignores typical_p
