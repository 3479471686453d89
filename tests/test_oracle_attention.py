"""Pins for the oracle's KV append, gather and decode attention (CPU only).

Each test checks the oracle against something other than itself: a hand-worked
golden fixture, a round trip, a library attention routine on contiguous K/V,
closed forms, or the split-softmax algebra.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _read_append_fixture(path):
    cfg, tables, lens, knew, vnew, expect = {}, {}, {}, {}, {}, []
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0] == "table":
            tables[int(f[1])] = [int(x) for x in f[2:]]
        elif f[0] == "seq_len":
            lens[int(f[1])] = int(f[2])
        elif f[0] in ("k_new", "v_new"):
            (knew if f[0] == "k_new" else vnew)[(int(f[1]), int(f[2]))] = [float(x) for x in f[3:]]
        elif f[0] == "expect":
            expect.append((f[1], int(f[2]), int(f[3]), int(f[4]), [float(x) for x in f[5:]]))
        else:
            cfg[f[0]] = int(f[1])
    return cfg, tables, lens, knew, vnew, expect


def test_append_golden_fixture(oracle_lib, golden_dir):
    cfg, tables, lens, knew, vnew, expect = _read_append_fixture(f"{golden_dir}/kv_append_small.txt")
    BS, NB, H, D = cfg["block_size"], cfg["num_blocks"], cfg["n_kv_heads"], cfg["head_dim"]
    B = len(lens)
    mb = max(len(t) for t in tables.values())
    bt = np.full((B, mb), -1, np.int32)
    for b, t in tables.items():
        bt[b, :len(t)] = t
    sl = np.array([lens[b] for b in range(B)], np.int32)
    kn = np.zeros((B, H, D), np.float32)
    vn = np.zeros((B, H, D), np.float32)
    for (b, h), v in knew.items():
        kn[b, h] = v
    for (b, h), v in vnew.items():
        vn[b, h] = v
    K = np.zeros((NB, H, BS, D), np.float32)
    V = np.zeros((NB, H, BS, D), np.float32)
    assert oracle_lib.kv_append(kn, vn, K, V, bt, sl, BS) == 0
    Kexp = np.zeros_like(K)
    Vexp = np.zeros_like(V)
    for which, blk, h, slot, vals in expect:
        (Kexp if which == "K" else Vexp)[blk, h, slot] = vals
    np.testing.assert_array_equal(K, Kexp)
    np.testing.assert_array_equal(V, Vexp)


def _build_pool_by_appends(oracle_lib, seqs_k, seqs_v, BS, NB, rng, dtype=np.float32):
    """Grow each sequence from empty by one oracle append per token (the lab's
    decode loop), with blocks handed out from a shuffled free list."""
    B = len(seqs_k)
    H, D = seqs_k[0].shape[1], seqs_k[0].shape[2]
    lens = [s.shape[0] for s in seqs_k]
    mb = max(-(-L // BS) for L in lens)
    free = list(rng.permutation(NB))
    bt = np.full((B, mb), -1, np.int32)
    K = np.zeros((NB, H, BS, D), dtype)
    V = np.zeros((NB, H, BS, D), dtype)
    for t in range(max(lens)):
        active = [b for b in range(B) if t < lens[b]]
        for b in active:
            if t % BS == 0:
                bt[b, t // BS] = free.pop()
        sl = np.array([t + 1 if t < lens[b] else 0 for b in range(B)], np.int32)
        kn = np.zeros((B, H, D), dtype)
        vn = np.zeros((B, H, D), dtype)
        for b in active:
            kn[b] = seqs_k[b][t]
            vn[b] = seqs_v[b][t]
        # sequences that are already finished pass L=0 and are reported/skipped
        st = oracle_lib.kv_append(kn, vn, K, V, bt, sl, BS)
        assert st in (0, 4)
    return K, V, bt, np.array(lens, np.int32)


def test_append_then_gather_round_trip(oracle_lib):
    """[LAB block 6] invariant: K/V gathered from scattered blocks equal the
    sequence that was appended, token by token, in order."""
    rng = np.random.default_rng(0)
    BS, NB, H, D = 4, 40, 3, 5
    lens = [1, 4, 5, 13, 22]
    sk = [rng.standard_normal((L, H, D)).astype(np.float32) for L in lens]
    sv = [rng.standard_normal((L, H, D)).astype(np.float32) for L in lens]
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, NB, rng)
    for b, L in enumerate(lens):
        for h in range(H):
            np.testing.assert_array_equal(oracle_lib.gather(K, bt, b, L, h), sk[b][:, h, :].astype(np.float64))
            np.testing.assert_array_equal(oracle_lib.gather(V, bt, b, L, h), sv[b][:, h, :].astype(np.float64))


def test_append_rejects_bad_length_and_block(oracle_lib):
    K = np.zeros((2, 1, 2, 1), np.float32)
    V = np.zeros_like(K)
    kn = np.ones((1, 1, 1), np.float32)
    bt = np.array([[0]], np.int32)
    assert oracle_lib.kv_append(kn, kn, K, V, bt, np.array([3], np.int32), 2) == 4  # beyond table
    assert oracle_lib.kv_append(kn, kn, K, V, bt, np.array([0], np.int32), 2) == 4  # nothing to append
    bt_bad = np.array([[7]], np.int32)
    assert oracle_lib.kv_append(kn, kn, K, V, bt_bad, np.array([1], np.int32), 2) == 4
    assert not K.any() and not V.any()


@pytest.mark.parametrize("G", [1, 2, 4])
def test_attention_matches_library_sdpa_on_contiguous_kv(oracle_lib, G):
    """[LAB block 5] cached attention equals full recompute: the oracle, reading K/V
    through the block table, matches torch's scaled_dot_product_attention in
    float64 on the contiguous K/V (GQA via the library's own enable_gqa)."""
    rng = np.random.default_rng(10 + G)
    BS, Hkv, D = 4, 2, 8
    Hq = Hkv * G
    lens = [1, 3, 4, 9, 17]
    NB = sum(-(-L // BS) for L in lens) + 5
    sk = [rng.standard_normal((L, Hkv, D)).astype(np.float32) for L in lens]
    sv = [rng.standard_normal((L, Hkv, D)).astype(np.float32) for L in lens]
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, NB, rng)
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float32)
    out, st, werr = oracle_lib.paged_attention(q, K, V, bt, sl)
    assert st == 0
    assert werr < 1e-12  # [LAB] asserts: attention weights sum to 1
    for b, L in enumerate(lens):
        qt = torch.from_numpy(q[b].astype(np.float64))[None, :, None, :]       # [1, Hq, 1, D]
        kt = torch.from_numpy(sk[b].astype(np.float64)).permute(1, 0, 2)[None]  # [1, Hkv, L, D]
        vt = torch.from_numpy(sv[b].astype(np.float64)).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, enable_gqa=True)
        np.testing.assert_allclose(out[b], ref[0, :, 0, :].numpy(), rtol=0, atol=1e-12)


def test_attention_closed_forms(oracle_lib):
    rng = np.random.default_rng(3)
    BS, Hkv, D, Hq = 2, 1, 4, 2
    # L = 1: the only weight is 1, output is V_0 exactly.
    sk = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    sv = [rng.standard_normal((1, Hkv, D)).astype(np.float32)]
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, 3, rng)
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    out, st, _ = oracle_lib.paged_attention(q, K, V, bt, sl)
    np.testing.assert_array_equal(out[0, 0], sv[0][0, 0].astype(np.float64))
    # All keys equal: uniform weights, output = mean of V.
    L = 7
    k_row = rng.standard_normal((1, Hkv, D)).astype(np.float32)
    sk = [np.repeat(k_row, L, axis=0)]
    sv = [rng.standard_normal((L, Hkv, D)).astype(np.float32)]
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, 6, rng)
    out, st, _ = oracle_lib.paged_attention(q, K, V, bt, sl)
    np.testing.assert_allclose(out[0, 1], sv[0][:, 0, :].astype(np.float64).mean(0), atol=1e-14)
    # One key far ahead of the rest: output is (numerically) that key's V row.
    sk = [rng.standard_normal((L, Hkv, D)).astype(np.float32)]
    qv = np.ones((1, Hq, D), np.float32)
    sk[0][4, 0, :] = 100.0
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, 6, rng)
    out, st, _ = oracle_lib.paged_attention(qv, K, V, bt, sl)
    np.testing.assert_allclose(out[0, 0], sv[0][4, 0, :].astype(np.float64), atol=1e-12)
    # L = 0: zeros.
    out, st, _ = oracle_lib.paged_attention(qv, K, V, bt, np.array([0], np.int32))
    assert st == 0 and not out.any()


def test_attention_scale_and_head_mapping(oracle_lib):
    """A scale override changes only the softmax temperature, and query head qh
    reads KV head qh // G: planting a huge key in KV head 1 moves only the
    outputs of query heads G..2G-1 ([CH5] 3.1 equal groups)."""
    rng = np.random.default_rng(4)
    BS, Hkv, D, G, L = 4, 2, 4, 3, 6
    sk = [rng.standard_normal((L, Hkv, D)).astype(np.float32)]
    sv = [rng.standard_normal((L, Hkv, D)).astype(np.float32)]
    sk[0][2, 1, :] = 50.0
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, 4, rng)
    q = np.ones((1, Hkv * G, D), np.float32)
    out, _, _ = oracle_lib.paged_attention(q, K, V, bt, sl)
    for qh in range(G, 2 * G):
        np.testing.assert_allclose(out[0, qh], sv[0][2, 1].astype(np.float64), atol=1e-12)
    for qh in range(G):
        assert np.abs(out[0, qh] - sv[0][2, 0]).max() > 1e-3
    # scale -> 0 makes every weight equal: the output is the mean of V.
    out0, _, _ = oracle_lib.paged_attention(q, K, V, bt, sl, scale=1e-300)
    np.testing.assert_allclose(out0[0, 0], sv[0][:, 0].astype(np.float64).mean(0), atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 4, 8, 12, 64])
def test_split_softmax_algebra_matches_two_pass(oracle_lib, chunk):
    """[CH5] 4.1: merging per-chunk (max, sum, unnormalised output) reproduces the
    two-pass softmax, for chunk sizes that cut blocks and the sequence tail."""
    rng = np.random.default_rng(chunk)
    BS, Hkv, D, Hq = 4, 2, 16, 4
    lens = [37, 50]
    sk = [rng.standard_normal((L, Hkv, D)).astype(np.float32) * 3 for L in lens]
    sv = [rng.standard_normal((L, Hkv, D)).astype(np.float32) for L in lens]
    K, V, bt, sl = _build_pool_by_appends(oracle_lib, sk, sv, BS, 40, rng)
    q = rng.standard_normal((2, Hq, D)).astype(np.float32)
    full, _, _ = oracle_lib.paged_attention(q, K, V, bt, sl)
    for b in range(2):
        for qh in range(Hq):
            sp = oracle_lib.attention_split_row(q, K, V, bt, sl, b, qh, chunk)
            np.testing.assert_allclose(sp, full[b, qh], rtol=0, atol=1e-12)


def test_attention_bf16_inputs_decode_exactly(oracle_lib):
    """bf16 inputs are the top 16 bits of float32: the oracle on bf16 bit patterns
    equals the oracle on the same values widened to float32."""
    rng = np.random.default_rng(5)
    BS, Hkv, D, Hq = 4, 1, 8, 2
    L = 11
    k32 = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    v32 = torch.from_numpy(rng.standard_normal((L, Hkv, D)).astype(np.float32)).to(torch.bfloat16)
    q16 = torch.from_numpy(rng.standard_normal((1, Hq, D)).astype(np.float32)).to(torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    Kb, Vb, bt, sl = _build_pool_by_appends(oracle_lib, [bits(k32)], [bits(v32)], BS, 5, rng, np.uint16)
    out_b, st, _ = oracle_lib.paged_attention(bits(q16), Kb, Vb, bt, sl)
    rng2 = np.random.default_rng(5)
    Kf, Vf, bt2, _ = _build_pool_by_appends(oracle_lib, [k32.float().numpy()], [v32.float().numpy()],
                                            BS, 5, np.random.default_rng(99))
    out_f, _, _ = oracle_lib.paged_attention(q16.float().numpy(), Kf, Vf, bt2, sl)
    np.testing.assert_allclose(out_b, out_f, rtol=0, atol=1e-15)


def test_attention_bad_inputs_give_zeros_and_status(oracle_lib):
    K = np.ones((2, 1, 2, 2), np.float32)
    q = np.ones((1, 1, 2), np.float32)
    out, st, _ = oracle_lib.paged_attention(q, K, K, np.array([[0]], np.int32), np.array([5], np.int32))
    assert st == 4 and not out.any()
    out, st, _ = oracle_lib.paged_attention(q, K, K, np.array([[9]], np.int32), np.array([1], np.int32))
    assert st == 4 and not out.any()
