"""GPU parity of chunked prefill: pkv_kv_append_chunk (whole pools bit-exact
against the oracle's append) and pkv_paged_prefill_attention (every row, or a
seeded sample at large sizes, against the float64 oracle within the bf16
tolerance 2e-2 / 2e-2).  Inputs: seeded chunk lengths (empty chunks, partial and
several 16-token tiles), cached prefixes of random length, one shuffled block
permutation, bf16 values; the slots past each sequence's end hold NaN, which
must not reach any output.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import TOL, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _inputs(seed, chunks, prefix_hi, Hq=32, Hkv=8, BS=16, D=128):
    rng = np.random.default_rng(seed)
    B = len(chunks)
    n = np.array(chunks, np.int64)
    prefix = rng.integers(0, prefix_hi + 1, B)
    L = (prefix + n).astype(np.int32)
    nb = (L + BS - 1) // BS
    MB = int(nb.max()) + 1
    NB = int(nb.sum()) + 3
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MB), -1, np.int32)
    o = 0
    for b in range(B):
        tables[b, :nb[b]] = perm[o:o + nb[b]]
        o += nb[b]
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    K = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda").to(torch.bfloat16)
    for b in range(B):                      # poison the slots past the end of every sequence
        if L[b] % BS:
            blk = int(tables[b, nb[b] - 1])
            K[blk, :, L[b] % BS:] = float("nan")
            V[blk, :, L[b] % BS:] = float("nan")
    T = int(n.sum())
    q_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    kn = torch.randn((T, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn((T, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((T, Hq, D), generator=g, device="cuda").to(torch.bfloat16)
    cu = lambda a: torch.from_numpy(a).cuda()
    return dict(K=K, V=V, kn=kn, vn=vn, q=q, tables=cu(tables), L=cu(L), q_start=cu(q_start), T=T, Hq=Hq)


def _check(inp, rows=None):
    Kh, Vh = host(inp["K"]), host(inp["V"])
    st = pkv.new_status()
    pkv.kv_append_chunk(inp["kn"], inp["vn"], inp["K"], inp["V"], inp["tables"], inp["L"], inp["q_start"], status=st)
    out = pkv.paged_prefill_attention(inp["q"], inp["K"], inp["V"], inp["tables"], inp["L"], inp["q_start"],
                                      status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    tb, L, qs = host(inp["tables"]), host(inp["L"]), host(inp["q_start"])
    assert oracle.kv_append_chunk(host(inp["kn"]), host(inp["vn"]), Kh, Vh, tb, L, qs) == oracle.OK
    np.testing.assert_array_equal(host(inp["K"]), Kh)
    np.testing.assert_array_equal(host(inp["V"]), Vh)
    ref, s2, werr = oracle.prefill_attention(host(inp["q"]), Kh, Vh, tb, L, qs, rows=rows)
    assert s2 == oracle.OK and werr < 1e-9
    got = out.float().cpu().numpy().reshape(-1, out.shape[-1])
    if rows is not None:
        got = got[np.asarray(rows)]
    assert np.isfinite(got).all()
    atol, rtol = TOL["bf16"]
    err = np.abs(got - ref)
    assert not (err > atol + rtol * np.abs(ref)).any(), float(err.max())
    return out


@pytest.mark.parametrize("chunks,prefix_hi,Hq,Hkv,BS", [
    ([1, 16, 37, 0, 100], 300, 32, 8, 16),
    ([5, 33], 2000, 64, 8, 16),     # 8 query heads per KV head
    ([17, 64, 3], 500, 8, 8, 32),   # one query head per KV head, 32-token blocks
    ([40, 7, 130], 700, 16, 8, 16),  # two query heads per KV head
    ([33, 90], 900, 24, 8, 16),      # three per KV head: 42 tokens x 3 heads per 128-row tile, 2 padding rows
    ([50, 20], 400, 56, 8, 16),      # seven per KV head: 18 tokens x 7 heads, 2 padding rows
    ([300, 129, 5], 600, 8, 8, 16),  # one per KV head, chunks filling both 128-token query tiles, ragged
])
def test_prefill_matches_oracle(chunks, prefix_hi, Hq, Hkv, BS):
    inp = _inputs(sum(chunks) + prefix_hi, chunks, prefix_hi, Hq=Hq, Hkv=Hkv, BS=BS)
    _check(inp)


@pytest.mark.parametrize("Hq,Hkv", [(24, 8), (32, 8)])
def test_prefill_unaligned_query_takes_the_mma_sync_kernel(Hq, Hkv):
    # q 8 bytes past a 16-byte boundary: the tensor-core kernel needs 16-byte
    # aligned rows, so the mma.sync kernel serves the call
    inp = _inputs(31, [40, 7, 130], 700, Hq=Hq, Hkv=Hkv)
    q = inp["q"]
    buf = torch.empty(q.numel() + 4, dtype=q.dtype, device=q.device)
    qu = buf[4:].view(q.shape)
    qu.copy_(q)
    assert qu.data_ptr() % 16 == 8
    inp["q"] = qu
    _check(inp)


def test_prefill_many_sequences():
    # 45 sequences: the CTAs' longest-first assignment walks the sequences 32 at a time
    rng = np.random.default_rng(17)
    chunks = [int(c) for c in rng.integers(0, 41, 45)]
    inp = _inputs(23, chunks, 700)
    _check(inp)


def test_prefill_long_chunks_sampled_rows():
    inp = _inputs(11, [512, 256, 1000, 128], 4000)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(inp["T"] * inp["Hq"], 400, replace=False))
    _check(inp, rows=rows)


def test_prefill_long_context_chunk():
    # a 4096-token chunk after a 12000-token prefix: key ranges past the
    # producers' 640-block table window, 64 chunk tiles of one sequence
    inp = _inputs(13, [4096, 3], 12000)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(inp["T"] * inp["Hq"], 400, replace=False))
    _check(inp, rows=rows)


def test_prefill_bad_length():
    inp = _inputs(4, [8, 8], 50)
    L = inp["L"].clone()
    L[1] = 5                               # shorter than its own 8-token chunk
    st = pkv.new_status()
    out = pkv.paged_prefill_attention(inp["q"], inp["K"], inp["V"], inp["tables"], L, inp["q_start"], status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 4
    assert (out[8:16].float() == 0).all()
