"""GPU parity of copy-on-write block sharing: pkv_copy_blocks against the
oracle's block copy (bit-exact, whole pools), and decode steps over forked
sequences that share prefix blocks, driven by the library's block pool.

Each step: the pool reserves every sequence's next slot (copy-on-write pairs
when a shared partial tail is written), pkv_copy_blocks copies them, kv_append
writes the new token, attention runs over the aliased tables.  The oracle
replays the copies and appends on host copies of the pools (whole pools must
match bit for bit) and recomputes attention in float64 over the same tables
(bf16 tolerance 2e-2 / 2e-2).  Invariant: attention over the aliased tables is
bit-identical to attention over the same sequences given private copies of
every block.
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


def _pools(NB, Hkv, BS, D, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    K = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda").to(dtype)
    V = torch.randn((NB, Hkv, BS, D), generator=g, device="cuda").to(dtype)
    return K, V


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_copy_blocks_bit_exact(dtype):
    NB, Hkv, BS, D = 300, 8, 16, 128
    K, V = _pools(NB, Hkv, BS, D, dtype, 11)
    Kh, Vh = host(K), host(V)
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(5))
    src, dst = perm[:100].to(torch.int32), perm[100:200].to(torch.int32)  # disjoint, distinct
    st = pkv.new_status()
    pkv.copy_blocks(K, V, src.cuda(), dst.cuda(), status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    assert oracle.copy_blocks(Kh, Vh, src.numpy(), dst.numpy()) == oracle.OK
    np.testing.assert_array_equal(host(K), Kh)
    np.testing.assert_array_equal(host(V), Vh)


def test_copy_blocks_odd_block_bytes_and_bad_ids():
    NB, Hkv, BS, D = 20, 3, 5, 7        # 210 bf16 per block: not a multiple of 16 bytes
    K, V = _pools(NB, Hkv, BS, D, torch.bfloat16, 12)
    Kh, Vh = host(K), host(V)
    src = torch.tensor([2, 50, 7], dtype=torch.int32)
    dst = torch.tensor([9, 3, -1], dtype=torch.int32)
    st = pkv.new_status()
    pkv.copy_blocks(K, V, src.cuda(), dst.cuda(), status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 4
    assert oracle.copy_blocks(Kh, Vh, src.numpy(), dst.numpy()) == oracle.DEVICE_BOUNDS
    np.testing.assert_array_equal(host(K), Kh)
    np.testing.assert_array_equal(host(V), Vh)
    pkv.copy_blocks(K, V, src[:0].cuda(), dst[:0].cuda())  # empty: no-op


def _attention_check(out, q, K, V, bt, sl):
    ref, _, werr = oracle.paged_attention(host(q), host(K), host(V), bt.numpy(), sl.numpy())
    assert werr < 1e-9
    got = out.float().cpu().numpy().reshape(ref.shape)
    atol, rtol = TOL["bf16"]
    err = np.abs(got - ref)
    assert not (err > atol + rtol * np.abs(ref)).any(), float(err.max())


@pytest.mark.parametrize("prompts,branches,lo,hi", [(4, 8, 100, 600), (2, 24, 1000, 3000)])
def test_forked_decode_steps(prompts, branches, lo, hi):
    Hq, Hkv, D, BS = 32, 8, 128, 16
    gen = torch.Generator().manual_seed(1000 + prompts)
    lens = torch.randint(lo, hi + 1, (prompts,), generator=gen).tolist()
    MB = (hi + 8) // BS + 2
    NB = sum(-(-L // BS) for L in lens) + prompts * branches * 2 + 8
    pool = pkv.BlockPool(NB, BS, MB)
    K, V = _pools(NB, Hkv, BS, D, torch.bfloat16, 2000 + prompts)  # prompt KV: whatever the blocks hold
    for p, L in enumerate(lens):
        pool.add(10_000 + p, L)
    children = []
    for p in range(prompts):
        for c in range(branches):
            cid = p * branches + c
            pool.fork(10_000 + p, cid)
            children.append(cid)
        pool.free(10_000 + p)           # the prompt itself retires; its blocks stay shared
    B = len(children)
    g = torch.Generator(device="cuda")
    g.manual_seed(3000 + prompts)
    Kh, Vh = host(K), host(V)
    st = pkv.new_status()
    n_cow = 0
    for step in range(3):
        pairs = [pool.append(s) for s in children]
        pairs = [p for p in pairs if p is not None]
        n_cow += len(pairs)
        bt, sl = pool.tables(children)
        if pairs:
            src = torch.tensor([p[0] for p in pairs], dtype=torch.int32)
            dst = torch.tensor([p[1] for p in pairs], dtype=torch.int32)
            pkv.copy_blocks(K, V, src.cuda(), dst.cuda(), status=st)
            oracle.copy_blocks(Kh, Vh, src.numpy(), dst.numpy())
        k_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        v_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        q = torch.randn((B, Hq, D), generator=g, device="cuda").to(torch.bfloat16)
        btd, sld = bt.cuda(), sl.cuda()
        pkv.kv_append(k_new, v_new, K, V, btd, sld, status=st)
        out = pkv.paged_decode_attention(q, K, V, btd, sld, status=st)
        torch.cuda.synchronize()
        assert pkv.check_status(st) == 0
        oracle.kv_append(host(k_new), host(v_new), Kh, Vh, bt.numpy(), sl.numpy(), BS)
        np.testing.assert_array_equal(host(K), Kh)
        np.testing.assert_array_equal(host(V), Vh)
        _attention_check(out, q, K, V, bt, sl)
    # step 0: of the branches sharing a partial tail, all but the last writer copy it
    assert n_cow == sum(branches - 1 for L in lens if L % BS)
    # aliasing invariant: private copies of every block give bit-identical output
    rows = []
    for i in range(B):
        n = -(-int(sl[i]) // BS)
        rows.append(bt[i, :n])
    flat = torch.cat(rows)
    NB2 = flat.numel()
    K2 = K[flat.cuda().long()].contiguous()
    V2 = V[flat.cuda().long()].contiguous()
    bt2 = torch.full_like(bt, -1)
    o = 0
    for i in range(B):
        n = rows[i].numel()
        bt2[i, :n] = torch.arange(o, o + n, dtype=torch.int32)
        o += n
    out2 = pkv.paged_decode_attention(q, K2, V2, bt2.cuda(), sld)
    torch.cuda.synchronize()
    assert NB2 > NB - pool.num_free()  # the private layout really holds more blocks
    assert torch.equal(out, out2)
