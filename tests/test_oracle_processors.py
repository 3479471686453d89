"""Pins of the oracle's logits processors (masks, penalties) and min-p (CPU).

"LLM inference serving tutorial" section 3.1 (pipeline order: hard
constraints, penalties, temperature, truncation filters), 3.2 (frequency /
presence penalty z - a_f c - a_p [c > 0]; sign-aware repetition penalty z / r
for z > 0, r z for z < 0, only on tokens that appeared), 3.3 (constrained
decoding: illegal logits set to -inf, then sampled as usual), Q4 and appendix
A [D01] (min-p keeps the most probable token; its support grows as min_p falls
and as T rises; adding a constant to every logit changes no support).  The
hand-worked processor example is tests/golden/logits_processor_example.txt.
"""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "logits_processor_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = [x.strip() for x in v.split(",")]
    return vals


def test_hand_worked_example():
    g = _golden()
    z = np.array([[float(x) for x in g["logits"]]], np.float32)
    mask = np.array([[int(g["mask_word"][0], 2)]], np.uint32)
    st = oracle.process_logits(z, mask=mask, row_ptr=[0, 3], tokens=[int(x) for x in g["tokens"]],
                               counts=[int(x) for x in g["counts"]], rep=[float(g["rep"][0])],
                               freq=[float(g["freq"][0])], pres=[float(g["pres"][0])])
    assert st == oracle.OK
    expect = np.array([[float(x) for x in g["expected"]]], np.float32)
    np.testing.assert_array_equal(z, expect)


def test_penalties_are_sign_aware_and_count_based():
    z = np.array([[2.0, -2.0, 0.0, 2.0, 2.0]], np.float32)
    oracle.process_logits(z, row_ptr=[0, 3], tokens=[0, 1, 2], counts=[1, 1, 1], rep=[1.5])
    assert z[0, 0] < 2.0 and z[0, 1] < -2.0 and z[0, 2] == 0.0   # not the same constant for every token
    assert math.isclose(z[0, 0], 2.0 / 1.5, rel_tol=1e-7) and math.isclose(z[0, 1], -3.0, rel_tol=1e-7)
    z = np.zeros((1, 4), np.float32)
    oracle.process_logits(z, row_ptr=[0, 3], tokens=[0, 1, 2], counts=[1, 2, 5], freq=[0.25], pres=[1.0])
    np.testing.assert_allclose(z[0], [-1.25, -1.5, -2.25, 0.0])  # linear in c, presence once, unlisted untouched
    z = np.zeros((1, 4), np.float32)
    oracle.process_logits(z, row_ptr=[0, 1], tokens=[3], counts=[0], freq=[1.0], pres=[1.0])
    assert (z == 0).all()                                          # c = 0: never appeared


def test_mask_then_sample_never_draws_a_banned_token():
    rng = np.random.default_rng(3)
    V = 70
    for s in range(40):
        z = rng.standard_normal((1, V)).astype(np.float32)
        allowed = rng.random(V) < 0.3
        allowed[rng.integers(V)] = True
        words = np.zeros((1, (V + 31) // 32), np.uint32)
        for i in np.flatnonzero(allowed):
            words[0, i // 32] |= np.uint32(1 << (i % 32))
        oracle.process_logits(z, mask=words)
        assert np.isneginf(z[0, ~allowed]).all() and np.isfinite(z[0, allowed]).all()
        r = oracle.sample_row(z[0], 1.0, 0, 0.9, s, 0)
        assert allowed[r["token"]]
    # a forced token: the only finite logit wins greedy and sampled draws
    z = rng.standard_normal((1, V)).astype(np.float32)
    words = np.zeros((1, 3), np.uint32)
    words[0, 1] = np.uint32(1 << 9)                                 # token 41
    oracle.process_logits(z, mask=words)
    assert oracle.sample_row(z[0], 0.0, 0, 1.0, 0, 0)["token"] == 41
    assert oracle.sample_row(z[0], 1.3, 5, 0.5, 7, 0)["token"] == 41


def test_min_p_support_d01():
    rng = np.random.default_rng(8)
    z = rng.standard_normal(64).astype(np.float32) * 2.0
    zmax = float(z.max())
    size = lambda T, a, zz=z: oracle.sample_row(zz, T, 0, 1.0, 1, 0, min_p=a)["n_kept"]
    for T in (0.2, 0.5, 1.0, 2.0, 5.0):
        for a in (0.05, 0.3, 0.9, 1.0):
            expect = int(np.sum(z.astype(np.float64) >= zmax + T * math.log(a)))   # closed form
            assert size(T, a) == expect and size(T, a) >= 1               # the maximum is always kept
    sizes = [size(T, 0.3) for T in (0.2, 0.5, 1.0, 2.0, 5.0)]
    assert sizes == sorted(sizes) and sizes[0] < sizes[-1]              # grows with T
    by_a = [size(1.0, a) for a in (0.9, 0.5, 0.2, 0.05, 0.01)]
    assert by_a == sorted(by_a)                                          # grows as min_p falls
    assert size(1.0, 0.3, z + np.float32(7.0)) == size(1.0, 0.3)         # shift invariance
    # draws stay in the support
    for s in range(50):
        t = oracle.sample_row(z, 1.0, 0, 1.0, s, 3, min_p=0.3)["token"]
        assert z[t] >= zmax + math.log(0.3)


def test_processor_and_min_p_errors():
    z = np.zeros((1, 8), np.float32)
    assert oracle.process_logits(z, row_ptr=[0, 1], tokens=[8], counts=[1], freq=[1.0]) == oracle.INVALID_ARG
    assert oracle.process_logits(z, row_ptr=[0, 1], tokens=[2], counts=[1], rep=[0.0]) == oracle.INVALID_ARG
    assert oracle.sample_row(z[0], 1.0, 0, 1.0, 0, 0, min_p=1.5)["status"] == oracle.INVALID_ARG
    assert oracle.sample_row(z[0], 1.0, 0, 1.0, 0, 0, min_p=float("nan"))["status"] == oracle.INVALID_ARG
