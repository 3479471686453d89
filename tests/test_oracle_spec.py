"""Pins of the speculative-verification oracle (oracle.spec_verify_row), CPU only.

Against what the pages and the mathematics fix ("Suy luan & Toi uu hoa
(Inference)" section 5.2 and exercise 5.5; "LLM inference serving tutorial"
section 7 / Q16): the worked example's acceptance rate alpha = sum min(p, q) =
0.78 (tests/golden/spec_verify_example.txt) by Monte Carlo, the distribution
preservation theorem (the emitted token follows p), the expected tokens per
cycle (1 - alpha^(gamma+1)) / (1 - alpha), the special cases q = p (every draft
kept, bonus token = the plain sampler's draw), disjoint supports (every draft
rejected, residual = p), greedy verification, the KV roll-back length, the
random stream (numpy's Philox), and the error cases.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "spec_verify_example.txt")


def _example():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = np.array([float(x) for x in v.split(",")])
    return vals["p"], vals["q"], float(vals["alpha"][0])


def _draft(q, rng):
    return int(rng.choice(len(q), p=q / q.sum()))


def test_alpha_of_the_worked_example():
    p, q, alpha = _example()
    assert abs(np.minimum(p, q).sum() - alpha) < 1e-12
    zt = np.log(np.stack([p, p])).astype(np.float32)
    zd = np.log(q)[None].astype(np.float32)
    rng = np.random.default_rng(5)
    n = 20000
    acc = 0
    first = np.zeros(len(p))
    for s in range(n):
        r = oracle.spec_verify_row(zt, zd, [_draft(q, rng)], 1.0, s, 0, 100)
        assert r["status"] == 0 and r["seq_len_out"] == 100 - 1 + r["n_acc"]
        acc += r["n_acc"]
        first[r["tokens"][0]] += 1
    sd = np.sqrt(alpha * (1 - alpha) / n)
    assert abs(acc / n - alpha) < 4.5 * sd
    # distribution preservation: the first emitted token follows p (chi-square, 5 dof)
    chi2 = float(((first - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 20.5, chi2   # 99.9% quantile of chi-square(5)


def test_expected_tokens_per_cycle():
    p, q, alpha = _example()
    gamma = 3
    zt = np.log(np.tile(p, (gamma + 1, 1))).astype(np.float32)
    zd = np.log(np.tile(q, (gamma, 1))).astype(np.float32)
    rng = np.random.default_rng(9)
    n = 12000
    emitted = [oracle.spec_verify_row(zt, zd, [_draft(q, rng) for _ in range(gamma)], 1.0, s, 7,
                                      50)["n_acc"] + 1 for s in range(n)]
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(np.mean(emitted) - expect) < 4.5 * np.std(emitted) / np.sqrt(n), (np.mean(emitted), expect)


def test_equal_distributions_keep_every_draft_and_bonus_is_the_sampler_draw():
    rng = np.random.default_rng(2)
    gamma, V = 4, 37
    for s in range(30):
        zt = rng.standard_normal((gamma + 1, V)).astype(np.float32)
        zd = zt[:gamma].copy()
        x = rng.integers(0, V, gamma).astype(np.int32)
        r = oracle.spec_verify_row(zt, zd, x, 0.8, s, 3, 20)
        assert r["n_acc"] == gamma and list(r["tokens"][:gamma]) == list(x)
        ref = oracle.sample_row(zt[gamma], 0.8, 0, 1.0, s, 3)
        assert r["tokens"][gamma] == ref["token"]
        assert r["seq_len_out"] == 20


def test_disjoint_supports_reject_and_draw_from_p():
    ninf = -np.inf
    zt = np.array([[0.0, np.log(3.0), ninf, ninf], [0.0, 0.0, 0.0, 0.0]], np.float32)  # p = (1/4, 3/4, 0, 0)
    zd = np.array([[ninf, ninf, 0.0, 0.0]], np.float32)                                 # q on {2, 3}
    n = 8000
    count0 = 0
    for s in range(n):
        r = oracle.spec_verify_row(zt, zd, [2 + (s & 1)], 1.0, s, 0, 9)
        assert r["n_acc"] == 0 and r["seq_len_out"] == 8 and r["tokens"][1] == -1
        assert r["tokens"][0] in (0, 1)
        count0 += r["tokens"][0] == 0
    assert abs(count0 / n - 0.25) < 4.5 * np.sqrt(0.25 * 0.75 / n)


def test_residual_is_max_of_p_minus_q():
    """p = (.5, .5, 0), q = (.5, 0, .5): a rejection happens only for x = 2, and the
    correction is then always token 1, where p exceeds q."""
    ninf = -np.inf
    zt = np.array([[0.0, 0.0, ninf], [0.0, 0.0, 0.0]], np.float32)
    zd = np.array([[0.0, ninf, 0.0]], np.float32)
    for s in range(200):
        r = oracle.spec_verify_row(zt, zd, [2], 1.0, s, 0, 5)
        assert r["n_acc"] == 0 and r["tokens"][0] == 1
        r = oracle.spec_verify_row(zt, zd, [0], 1.0, s, 0, 5)   # p/q = 1 at x = 0: kept
        assert r["n_acc"] == 1 and r["tokens"][0] == 0


def test_greedy_verification():
    rng = np.random.default_rng(4)
    gamma, V = 5, 50
    zt = rng.standard_normal((gamma + 1, V)).astype(np.float32)
    zd = rng.standard_normal((gamma, V)).astype(np.float32)
    am = zt.argmax(axis=1)
    for k in range(gamma + 1):
        x = am[:gamma].copy()
        if k < gamma:
            x[k] = (x[k] + 1) % V
        r = oracle.spec_verify_row(zt, zd, x.astype(np.int32), 0.0, 1, 1, 30)
        assert r["n_acc"] == k
        assert list(r["tokens"][:k]) == list(x[:k]) and r["tokens"][k] == am[k]
        assert all(t == -1 for t in r["tokens"][k + 1:])
        assert r["seq_len_out"] == 30 - gamma + k


def test_stream_counters_match_numpy_philox():
    """Uniform number j is numpy's Philox at counter (offset, j, 0, 0) - 1 in its
    first word (numpy advances the counter before its first block)."""
    for seed, off, j in [(0, 0, 0), (5, 7, 1), (2**63 + 11, 2**40, 4), (123, 0, 31)]:
        c = (off + (j << 64) - 1) % 2**256          # the 256-bit counter minus one
        ctr = np.array([(c >> (64 * w)) & (2**64 - 1) for w in range(4)], dtype=np.uint64)
        word = np.random.Philox(key=np.array([seed, 0], np.uint64), counter=ctr).random_raw(1)[0]
        assert oracle.uniform_at(seed, off, j) == int(word >> np.uint64(11)) * 2.0**-53
    assert oracle.uniform_at(9, 4, 0) == oracle.uniform(9, 4)


def test_error_cases():
    zt = np.zeros((2, 4), np.float32)
    zd = np.zeros((1, 4), np.float32)
    assert oracle.spec_verify_row(zt, zd, [4], 1.0, 0, 0, 5)["status"] == oracle.INVALID_ARG
    assert oracle.spec_verify_row(zt, zd, [1], -1.0, 0, 0, 5)["status"] == oracle.INVALID_ARG
    assert oracle.spec_verify_row(zt, zd, [1], 1.0, 0, 0, 0)["status"] == oracle.INVALID_ARG
    bad = zt.copy()
    bad[1, 2] = np.nan
    r = oracle.spec_verify_row(bad, zd, [1], 1.0, 0, 0, 5)
    assert r["status"] == oracle.NONFINITE and list(r["tokens"]) == [-1, -1] and r["seq_len_out"] == 5
    allinf = np.full((2, 4), -np.inf, np.float32)
    assert oracle.spec_verify_row(allinf, zd, [1], 1.0, 0, 0, 5)["status"] == oracle.NONFINITE
    # gamma = 0: a plain draw from p_1
    r = oracle.spec_verify_row(zt[:1], np.zeros((0, 4), np.float32), np.zeros(0, np.int32), 1.0, 3, 2, 7)
    assert r["n_acc"] == 0 and r["seq_len_out"] == 7
    assert r["tokens"][0] == oracle.sample_row(zt[0], 1.0, 0, 1.0, 3, 2)["token"]
