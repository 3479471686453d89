"""Pins for the oracle's sampler and Philox stream (CPU only).

Pins used: the pages' worked support sets ([D01]/[D02] and the nucleus
definition), brute-force enumeration of every candidate support on tiny
vocabularies, closed-form special cases (k=1, p->0, T->0, greedy ties, shift
invariance), numpy's own Philox4x64 for the random stream, and a chi-square test
that draws follow the renormalised distribution.
"""
import itertools
import math

import numpy as np
import pytest


def _support(probs):
    return {i for i, p in enumerate(probs) if p > 0}


def _load_examples(path):
    rows = []
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        name, probs, k, p, sup = line.split()
        rows.append((name, [float(x) for x in probs.split(",")], int(k), float(p),
                     {int(x) for x in sup.split(",")}))
    return rows


def test_worked_support_examples(oracle_lib, golden_dir):
    for name, probs, k, p, expected in _load_examples(f"{golden_dir}/sampler_support_examples.txt"):
        z = np.log(np.array(probs, np.float64)).astype(np.float32)
        r = oracle_lib.sample_row(z, 1.0, k, p, seed=1, offset=0, want_probs=True)
        assert r["status"] == 0, name
        assert _support(r["probs"]) == expected, name
        assert abs(r["probs"].sum() - 1.0) < 1e-12, name           # [LAB] probabilities sum to 1
        assert r["token"] in expected, name


def test_filter_order_is_topk_then_topp(oracle_lib):
    """[D02]: top-k then top-p gives {0,1}; the reverse order would give {0,1,2},
    which the fixed pipeline must not produce."""
    z = np.log(np.array([0.5, 0.2, 0.15, 0.1, 0.05])).astype(np.float32)
    r = oracle_lib.sample_row(z, 1.0, 3, 0.8, 0, 0, want_probs=True)
    assert _support(r["probs"]) == {0, 1}
    assert _support(r["probs"]) != {0, 1, 2}


def _brute_force_support(z, T, k, p):
    """Smallest 'upper set' (closed under the (-z, id) order) satisfying the
    definitions, found by enumerating every subset of the vocabulary."""
    V = len(z)
    fin = [i for i in range(V) if np.isfinite(z[i])]
    rank = lambda i: (-float(z[i]), i)
    def upward_closed(S, universe):
        return all(rank(i) < rank(j) for i in S for j in universe if j not in S)
    kk = len(fin) if (k <= 0 or k >= len(fin)) else k
    topk = None
    for S in itertools.combinations(fin, kk):
        if upward_closed(set(S), fin):
            topk = set(S)
            break
    zmax = max(float(z[i]) for i in topk)
    w = {i: math.exp((float(z[i]) - zmax) / T) for i in topk}
    Z = sum(w.values())
    if p >= 1.0:
        return topk, {i: w[i] / Z for i in topk}
    best = None
    for size in range(1, len(topk) + 1):
        for S in itertools.combinations(sorted(topk), size):
            S = set(S)
            if upward_closed(S, topk) and sum(w[i] for i in S) / Z >= p:
                best = S
                break
        if best is not None:
            break
    Zp = sum(w[i] for i in best)
    return best, {i: w[i] / Zp for i in best}


@pytest.mark.parametrize("trial", range(40))
def test_brute_force_tiny_vocab(oracle_lib, trial):
    rng = np.random.default_rng(trial)
    V = int(rng.integers(1, 9))
    z = rng.integers(-3, 4, V).astype(np.float32) * 0.5  # small integers -> many ties
    if V > 2 and trial % 3 == 0:
        z[rng.integers(0, V)] = -np.inf                   # a banned token
    if not np.isfinite(z).any():
        z[0] = 0.0
    # the sampler's temperature and top_p are float32 parameters
    T = float(np.float32(rng.choice([0.3, 0.7, 1.0, 2.5])))
    k = int(rng.integers(0, V + 2))
    p = float(np.float32(rng.choice([0.05, 0.3, 0.5, 0.77, 0.9, 1.0])))
    exp_sup, exp_probs = _brute_force_support(z, T, k, p)
    r = oracle_lib.sample_row(z, T, k, p, seed=trial, offset=3, want_probs=True)
    assert r["status"] == 0
    # the brute force uses float exp/sum; exact cut ties within 1e-12 are skipped
    if r["cut_margin"] > 1e-12:
        assert _support(r["probs"]) == exp_sup
        for i, pi in exp_probs.items():
            assert abs(r["probs"][i] - pi) < 1e-12
    assert r["token"] in _support(r["probs"])


def test_special_cases(oracle_lib):
    rng = np.random.default_rng(7)
    z = rng.standard_normal(1000).astype(np.float32) * 2
    am = int(np.argmax(z))
    for seed in range(20):
        assert oracle_lib.sample_row(z, 0.8, 1, 1.0, seed, 0)["token"] == am      # k = 1
        assert oracle_lib.sample_row(z, 0.8, 0, 1e-9, seed, 0)["token"] == am    # p -> 0+
        assert oracle_lib.sample_row(z, 1e-4, 0, 1.0, seed, 0)["token"] == am    # T -> 0+ ([D01])
        assert oracle_lib.sample_row(z, 0.0, 50, 0.5, seed, 0)["token"] == am    # greedy branch
    # greedy picks the lowest index among tied maxima ([SERVE] 3.1)
    zt = np.array([1.0, 3.0, -np.inf, 3.0, 2.0], np.float32)
    assert oracle_lib.sample_row(zt, 0.0, 0, 1.0, 0, 0)["token"] == 1
    # T -> 0+ with a tied maximum splits the mass evenly ([D01])
    r = oracle_lib.sample_row(zt, 1e-3, 0, 1.0, 0, 0, want_probs=True)
    assert _support(r["probs"]) == {1, 3} and abs(r["probs"][1] - 0.5) < 1e-12
    # adding a constant to every logit changes neither support nor token ([D01])
    for seed in range(20):
        a = oracle_lib.sample_row(z, 0.9, 50, 0.8, seed, 5, want_probs=True)
        b = oracle_lib.sample_row(z + np.float32(4.0), 0.9, 50, 0.8, seed, 5, want_probs=True)
        assert a["token"] == b["token"] and _support(a["probs"]) == _support(b["probs"])
    # top-k support has exactly k tokens when logits are distinct ([D01])
    for k in (1, 7, 100):
        assert oracle_lib.sample_row(z, 1.3, k, 1.0, 0, 0)["n_kept"] == k
    # -0.0 and +0.0 are the same logit: ties fall back to the token id
    zz = np.array([0.0, -0.0, -1.0], np.float32)
    r = oracle_lib.sample_row(zz, 1.0, 1, 1.0, 0, 0, want_probs=True)
    assert _support(r["probs"]) == {0}
    zz = np.array([-0.0, 0.0, -1.0], np.float32)
    r = oracle_lib.sample_row(zz, 1.0, 1, 1.0, 0, 0, want_probs=True)
    assert _support(r["probs"]) == {0}


def test_error_cases(oracle_lib):
    z = np.zeros(4, np.float32)
    assert oracle_lib.sample_row(z, -1.0, 0, 1.0, 0, 0)["status"] == 1         # T < 0 rejected
    assert oracle_lib.sample_row(z, 1.0, 0, 0.0, 0, 0)["status"] == 1          # p <= 0
    zn = z.copy(); zn[2] = np.nan
    r = oracle_lib.sample_row(zn, 1.0, 0, 1.0, 0, 0)
    assert r["status"] == 6 and r["token"] == -1
    zi = np.full(4, -np.inf, np.float32)
    assert oracle_lib.sample_row(zi, 1.0, 0, 1.0, 0, 0)["status"] == 6        # all banned
    zp = z.copy(); zp[1] = np.inf
    assert oracle_lib.sample_row(zp, 1.0, 0, 1.0, 0, 0)["status"] == 6


def test_philox_matches_numpy(oracle_lib):
    """Philox4x64-10 against numpy's implementation (numpy advances the counter
    once before producing its first block)."""
    rng = np.random.default_rng(11)
    for _ in range(50):
        key = rng.integers(0, 2**64, 2, dtype=np.uint64)
        ctr = rng.integers(0, 2**64, 4, dtype=np.uint64)
        ctr[0] = ctr[0] if ctr[0] != np.uint64(2**64 - 1) else np.uint64(0)
        ref = np.random.Philox(key=key, counter=ctr).random_raw(4)
        mine_ctr = ctr.copy()
        mine_ctr[0] = mine_ctr[0] + np.uint64(1)
        np.testing.assert_array_equal(oracle_lib.philox4x64_10(mine_ctr, key), ref)


def test_uniform_and_inverse_cdf_against_numpy_stream(oracle_lib):
    """Two tokens at 0.25 / 0.75: the draw is token 0 exactly when the uniform
    (top 53 bits of numpy's Philox word 0, times 2^-53) is below 0.25."""
    z = np.log(np.array([0.25, 0.75])).astype(np.float32)
    zero = np.zeros(4, dtype=np.uint64)
    for seed in range(200):
        ctr = zero.copy()
        ctr[0] = np.uint64(2**64 - 1)  # so that numpy's first block uses counter 0
        ctr[1] = np.uint64(2**64 - 1); ctr[2] = np.uint64(2**64 - 1); ctr[3] = np.uint64(2**64 - 1)
        word = np.random.Philox(key=np.array([seed, 0], np.uint64), counter=ctr).random_raw(1)[0]
        u = int(word >> np.uint64(11)) * 2.0**-53
        assert abs(oracle_lib.uniform(seed, 0) - u) == 0.0
        r = oracle_lib.sample_row(z, 1.0, 0, 1.0, seed, 0, want_probs=True)
        cut = r["probs"][0]
        if abs(u - cut) > 1e-12:
            assert r["token"] == (0 if u < cut else 1)


def test_draws_follow_renormalised_distribution(oracle_lib):
    """Chi-square: 20000 draws (offsets 0..19999) against the final distribution."""
    z = np.array([1.2, 0.3, -0.4, 2.0, 0.9, -1.5, 0.0, 0.5], np.float32)
    T, k, p = 0.9, 6, 0.9
    probs = oracle_lib.sample_row(z, T, k, p, 0, 0, want_probs=True)["probs"]
    n = 20000
    logits = np.tile(z, (n, 1))
    res = oracle_lib.sample_batch(logits, np.full(n, T), np.full(n, k), np.full(n, p),
                                  np.full(n, 12345, np.uint64), np.arange(n, dtype=np.uint64))
    counts = np.bincount(res["tokens"], minlength=len(z))
    sup = probs > 0
    assert (counts[~sup] == 0).all()
    exp = probs[sup] * n
    chi2 = float(((counts[sup] - exp) ** 2 / exp).sum())
    dof = int(sup.sum()) - 1
    # 99.9% quantile of chi-square with dof <= 7 is below 24.4
    assert chi2 < 24.4, (chi2, dof)
    # independent requests: different seeds at the same offset also match
    res2 = oracle_lib.sample_batch(logits, np.full(n, T), np.full(n, k), np.full(n, p),
                                   np.arange(n, dtype=np.uint64), np.zeros(n, np.uint64))
    counts2 = np.bincount(res2["tokens"], minlength=len(z))
    chi2b = float(((counts2[sup] - exp) ** 2 / exp).sum())
    assert chi2b < 24.4
