"""Pins of the chunked-prefill oracle (oracle.kv_append_chunk, oracle.prefill_attention), CPU.

Against a library routine and invariants ("Suy luan & Toi uu hoa (Inference)"
2.1 and the lab's chunked prefill: the chunk's token i sits at position
L - n + i and attends to every position up to its own):
* torch's scaled_dot_product_attention in float64 with an explicit causal mask
  over contiguous per-sequence K/V (built before they are scattered into the
  paged pool), with GQA heads expanded;
* a one-token chunk equals the decode attention of the same step;
* a chunk of n tokens equals n one-token steps appended in turn;
* after the chunk append, reading a sequence through its table gives the old
  prefix followed by the new rows.
"""
import numpy as np
import pytest
import torch

import oracle


def _case(seed, B=3, Hq=4, Hkv=2, D=8, BS=4, lo=1, hi=19, dtype=np.float32):
    rng = np.random.default_rng(seed)
    n = rng.integers(1, 7, B)                       # new tokens per sequence
    L = np.array([rng.integers(max(lo, k), hi + 1) for k in n])   # lengths after the chunk
    nb = (L + BS - 1) // BS
    NB = int(nb.sum()) + 5
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, int(nb.max())), -1, np.int32)
    o = 0
    for b in range(B):
        tables[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    Kc = [rng.standard_normal((L[b], Hkv, D)) for b in range(B)]     # contiguous K/V, whole sequences
    Vc = [rng.standard_normal((L[b], Hkv, D)) for b in range(B)]
    Kp = rng.standard_normal((NB, Hkv, BS, D)).astype(dtype)           # garbage everywhere else
    Vp = rng.standard_normal((NB, Hkv, BS, D)).astype(dtype)
    for b in range(B):                              # the prefix (all but the chunk) already cached
        for pos in range(L[b] - n[b]):
            Kp[tables[b, pos // BS], :, pos % BS] = Kc[b][pos]
            Vp[tables[b, pos // BS], :, pos % BS] = Vc[b][pos]
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    kn = np.concatenate([Kc[b][L[b] - n[b]:] for b in range(B)]).astype(dtype)
    vn = np.concatenate([Vc[b][L[b] - n[b]:] for b in range(B)]).astype(dtype)
    q = rng.standard_normal((int(q_start[-1]), Hq, D)).astype(dtype)
    return dict(n=n, L=L.astype(np.int32), tables=tables, Kp=Kp, Vp=Vp, Kc=Kc, Vc=Vc, q_start=q_start, kn=kn,
                vn=vn, q=q, BS=BS, Hq=Hq, Hkv=Hkv, D=D)


def test_chunk_append_then_gather_is_prefix_plus_rows():
    c = _case(1)
    st = oracle.kv_append_chunk(c["kn"], c["vn"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    assert st == oracle.OK
    for b in range(len(c["L"])):
        for h in range(c["Hkv"]):
            got = oracle.gather(c["Kp"], c["tables"], b, int(c["L"][b]), h)
            np.testing.assert_array_equal(got, c["Kc"][b][:, h].astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("seed", [2, 3, 4])
def test_causal_chunk_attention_matches_sdpa(seed):
    c = _case(seed)
    oracle.kv_append_chunk(c["kn"], c["vn"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    out, st, werr = oracle.prefill_attention(c["q"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    assert st == oracle.OK and werr < 1e-12
    out = out.reshape(-1, c["Hq"], c["D"])
    G = c["Hq"] // c["Hkv"]
    for b in range(len(c["L"])):
        L, n = int(c["L"][b]), int(c["n"][b])
        K = torch.tensor(c["Kc"][b].astype(np.float32), dtype=torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
        V = torch.tensor(c["Vc"][b].astype(np.float32), dtype=torch.float64).permute(1, 0, 2).repeat_interleave(G, 0)
        qb = torch.tensor(c["q"][c["q_start"][b]:c["q_start"][b + 1]], dtype=torch.float64).permute(1, 0, 2)
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]       # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(qb, K, V, attn_mask=mask)  # [Hq, n, D]
        np.testing.assert_allclose(out[c["q_start"][b]:c["q_start"][b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def test_one_token_chunk_is_the_decode_step():
    c = _case(5)
    # keep only the last new token of each sequence as a one-token chunk
    oracle.kv_append_chunk(c["kn"], c["vn"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    last = c["q_start"][1:] - 1
    q1 = np.ascontiguousarray(c["q"][last])
    out_p, st, _ = oracle.prefill_attention(q1, c["Kp"], c["Vp"], c["tables"], c["L"],
                                            np.arange(len(c["L"]) + 1, dtype=np.int32))
    out_d, st2, _ = oracle.paged_attention(q1, c["Kp"], c["Vp"], c["tables"], c["L"])
    assert st == st2 == oracle.OK
    np.testing.assert_array_equal(out_p.reshape(out_d.shape), out_d)


def test_chunk_equals_sequential_steps():
    c = _case(6)
    full = c["Kp"].copy(), c["Vp"].copy()
    oracle.kv_append_chunk(c["kn"], c["vn"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    ref, _, _ = oracle.prefill_attention(c["q"], c["Kp"], c["Vp"], c["tables"], c["L"], c["q_start"])
    Kp, Vp = full
    B = len(c["L"])
    for b in range(B):
        n, L = int(c["n"][b]), int(c["L"][b])
        for i in range(n):
            t = int(c["q_start"][b]) + i
            sl = np.array([L - n + i + 1], np.int32)
            qs = np.array([0, 1], np.int32)
            tb = c["tables"][b:b + 1]
            oracle.kv_append_chunk(c["kn"][t:t + 1], c["vn"][t:t + 1], Kp, Vp, tb, sl, qs)
            o, st, _ = oracle.prefill_attention(np.ascontiguousarray(c["q"][t:t + 1]), Kp, Vp, tb, sl, qs)
            assert st == oracle.OK
            np.testing.assert_allclose(o, ref[t * c["Hq"]:(t + 1) * c["Hq"]], rtol=0, atol=1e-13)


def test_chunk_errors():
    c = _case(7)
    bad = c["L"].copy()
    bad[1] = int(c["n"][1]) - 1            # shorter than its own chunk
    assert oracle.kv_append_chunk(c["kn"], c["vn"], c["Kp"], c["Vp"], c["tables"], bad,
                                  c["q_start"]) == oracle.DEVICE_BOUNDS
    _, st, _ = oracle.prefill_attention(c["q"], c["Kp"], c["Vp"], c["tables"], bad, c["q_start"])
    assert st == oracle.DEVICE_BOUNDS
