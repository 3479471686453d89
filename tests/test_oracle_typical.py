"""Pins of the typical-sampling oracle (oracle.sample_row_typical), CPU.

"LLM inference serving tutorial" section 3.1 (other samplers) defines typical
sampling: H(p) = -sum p ln p, d_i = |-ln p_i - H|, keep the smallest prefix in
ascending d whose cumulative probability reaches typical_p, renormalise.  Pinned
to the page's worked example ([D01], tests/golden/typical_sampling_d01.txt),
closed forms (uniform rows: H = ln n, every d = 0, so the first ceil(tau n) ids
are kept), the interval property of the kept set, shift invariance, the
typical_p >= 1 and T = 0 reductions to the pinned sampler, the literal
float64 definition on well-separated rows, and a chi-square test of the draws.
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
    # (up to the 2^-8 rounding of the centre and float32 rounding)
    assert dist[~kept].min() >= dist[kept].max() - 2 * 2.0**-9 - 1e-5
    # the kept mass reaches typical_p, and dropping one of the farthest kept
    # tokens (those within the rounding band of the boundary) would not
    assert p[kept].sum() >= np.float32(tp) - 1e-12
    band = np.nonzero(kept & (dist >= dist[kept].max() - 2.0**-8 - 1e-5))[0]
    assert any(p[kept].sum() - p[j] < np.float32(tp) + 1e-9 for j in band)
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


def test_literal_definition_on_separated_rows():
    """Where no two tokens are close in d and the centre is far from a
    rounding midpoint, the float32 order equals the literal float64 order."""
    checked = 0
    for seed in range(200):
        rng = np.random.default_rng(200 + seed)
        V = int(rng.integers(4, 9))
        z = (rng.standard_normal(V) * 1.5).astype(np.float32)
        T = 1.0
        p = np.exp((z.astype(np.float64) - z.max()) / T)
        p /= p.sum()
        H = float(-(p * np.log(p)).sum())
        d = np.abs(-np.log(p) - H)
        if np.diff(np.sort(d)).min() < 1e-3 or oracle.sample_row_typical(z, T, 0.5, 1, 0)["center_margin"] < 1e-4:
            continue
        order = sorted(range(V), key=lambda i: (d[i], -p[i], i))
        for tp in (0.1, 0.3, 0.5, 0.7, 0.9):
            cum, keep = 0.0, set()
            for i in order:
                keep.add(i)
                cum += p[i]
                if cum >= np.float32(tp):
                    break
            r = oracle.sample_row_typical(z, T, tp, 1, 0, want_probs=True)
            assert _support(r) == keep, (seed, tp)
        checked += 1
        if checked == 12:
            break
    assert checked == 12


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
