"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small and medium shapes that span several tiles, CTA ranges and ragged tails,
plus the decode-step edge cases.  Full-size workloads are in test_gpu_full.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from paged_kv_decode_table_gb300 import workloads as W
from tests.gpu_helpers import compare_attention, compare_tokens, host, run_attention, sampler_args

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    oracle.build()


# ----------------------------------------------------------------- kv_append
@pytest.mark.parametrize("num,over", [(1, {}), (4, dict(batch=37)), (2, dict(batch=9, len_lo=1, len_hi=900))])
def test_kv_append_bit_exact(num, over):
    w = W.workload(num, **over)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    Kh, Vh = host(inp["k_cache"]), host(inp["v_cache"])
    st = pkv.new_status()
    pkv.kv_append(inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                  inp["seq_lens"], status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    assert oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), Kh, Vh, host(inp["block_tables"]),
                            host(inp["seq_lens"]), w.block_size) == 0
    # whole pools compared bit for bit: catches stray writes anywhere
    np.testing.assert_array_equal(host(inp["k_cache"]), Kh)
    np.testing.assert_array_equal(host(inp["v_cache"]), Vh)


def test_kv_append_bad_rows_are_skipped_and_reported():
    w = W.workload(2, batch=6, len_lo=100, len_hi=600)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    sl = inp["seq_lens"].clone()
    sl[1] = 0                                   # nothing to append
    sl[2] = w.max_blocks * w.block_size + 1     # beyond the table
    bt = inp["block_tables"].clone()
    bt[3, (int(sl[3]) - 1) // w.block_size] = inp["num_blocks"] + 5   # bad block id
    Kh, Vh = host(inp["k_cache"]), host(inp["v_cache"])
    st = pkv.new_status()
    pkv.kv_append(inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], bt, sl, status=st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 4
    assert oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), Kh, Vh, host(bt), host(sl),
                            w.block_size) == 4
    np.testing.assert_array_equal(host(inp["k_cache"]), Kh)
    np.testing.assert_array_equal(host(inp["v_cache"]), Vh)


# ----------------------------------------------------------------- attention
CASES = [
    # (workload, overrides, label)
    (1, {}, "tiny-lab-f32 (generic kernel)"),
    (2, dict(batch=5, len_lo=1, len_hi=700), "gqa-G4 ragged (fast kernel)"),
    (2, dict(batch=40, len_lo=16, len_hi=300), "gqa-G4 many short (fast kernel)"),
    (3, dict(batch=3, len_lo=3000, len_hi=9000), "gqa-G8 long (fast kernel, split)"),
    (4, dict(batch=64), "fragmented pool with holes (fast kernel)"),
    (2, dict(batch=6, head_dim=64, len_lo=1, len_hi=400), "bf16 D=64 (generic kernel)"),
    (2, dict(batch=4, n_q_heads=48, n_kv_heads=4, len_lo=100, len_hi=500), "G=12 rows>8 (fast kernel)"),
    (2, dict(batch=4, n_q_heads=8, n_kv_heads=8, len_lo=100, len_hi=500), "MHA G=1 (fast kernel)"),
    (2, dict(batch=4, block_size=32, n_kv_heads=4, n_q_heads=16, len_lo=33, len_hi=700), "block_size 32 (fast kernel)"),
    (2, dict(batch=4, dtype="f32", len_lo=1, len_hi=300), "f32 D=128 (generic kernel)"),
    (3, dict(batch=1, len_lo=262144, len_hi=262144), "one 256K-token sequence split over every SM (fast kernel)"),
    (2, dict(batch=2048, len_lo=1, len_hi=48), "2048 short sequences, many per range (fast kernel)"),
]


@pytest.mark.parametrize("num,over,label", CASES, ids=[c[2] for c in CASES])
def test_attention_parity(num, over, label):
    w = W.workload(num, **over)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    st = pkv.new_status()
    out = run_attention(inp, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    err, n = compare_attention(out, inp, w.dtype)
    print(f"{label}: max |err| {err:.3e} over {n} rows")


def test_attention_poisoned_tails_and_edge_lengths():
    """Slots past each sequence's end hold NaN: they must never reach the output.
    Lengths 0, 1, exact block multiples and the table maximum are all present."""
    w = W.workload(2, batch=8, len_lo=200, len_hi=256)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    BS, mb = w.block_size, w.max_blocks
    lens = [0, 1, 16, 17, 255, 256, mb * BS, 33]
    # rebuild tables for these lengths over the same pool
    need = [-(-L // BS) for L in lens]
    perm = torch.randperm(inp["num_blocks"], generator=torch.Generator().manual_seed(5))
    assert sum(need) <= inp["num_blocks"]
    bt = torch.full((w.batch, mb), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    inp["block_tables"] = bt.cuda()
    inp["seq_lens"] = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for b, L in enumerate(lens):
        if L % BS:
            blk = int(bt[b, L // BS])
            inp["k_cache"][blk, :, L % BS:, :] = float("nan")
            inp["v_cache"][blk, :, L % BS:, :] = float("nan")
    st = pkv.new_status()
    out = run_attention(inp, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    assert torch.isfinite(out.float()).all()
    assert (out[0] == 0).all()          # L = 0 -> zeros
    compare_attention(out, inp, "bf16")


@pytest.mark.parametrize("num,over", [(2, dict(batch=6, len_lo=100, len_hi=600)), (1, {})])
def test_attention_bad_inputs_give_zero_rows_and_status(num, over):
    w = W.workload(num, **over)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    sl = inp["seq_lens"].clone()
    bt = inp["block_tables"].clone()
    sl[0] = w.max_blocks * w.block_size + 3            # length beyond the table
    bt[1, 0] = -7                                       # bad block id inside the sequence
    inp["seq_lens"], inp["block_tables"] = sl, bt
    st = pkv.new_status()
    out = run_attention(inp, st)
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 4
    assert (out[0] == 0).all() and (out[1] == 0).all()
    if w.batch > 2:
        rows = np.arange(2 * w.n_q_heads, w.batch * w.n_q_heads)
        # untouched sequences are still correct
        got = out.float().cpu().numpy().reshape(-1, w.head_dim)[rows]
        ref, _, _ = oracle.paged_attention(host(inp["q"]), host(inp["k_cache"]), host(inp["v_cache"]),
                                           host(bt), host(sl), rows=rows)
        assert np.abs(got - ref).max() < 2e-2


def test_attention_deterministic_and_scale_override():
    w = W.workload(3, batch=2, len_lo=2000, len_hi=5000)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    a = run_attention(inp).clone()
    b = run_attention(inp)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    out = pkv.paged_decode_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                                     inp["seq_lens"], scale=0.05)
    ref, _, _ = oracle.paged_attention(host(inp["q"]), host(inp["k_cache"]), host(inp["v_cache"]),
                                       host(inp["block_tables"]), host(inp["seq_lens"]), scale=0.05)
    got = out.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2e-2 + 2e-2 * np.abs(ref))


def test_attention_workspace_contents_and_graph_replay():
    """The workspace's contents are ignored on entry: the result must not
    depend on what it held before (random bytes, or what a previous call left),
    and replays of one captured launch must match the eager call bit for bit."""
    w = W.workload(2, batch=24)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    args = (inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["seq_lens"])
    nbytes = pkv.decode_workspace_bytes(w.batch, w.n_q_heads, w.head_dim)
    ws0 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ref = pkv.paged_decode_attention(*args, workspace=ws0).clone()
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    wsr = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    for _ in range(3):
        pkv.paged_decode_attention(*args, out=out, workspace=wsr)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    st = pkv.new_status()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkv.paged_decode_attention(*args, out=out, workspace=wsr, status=st)   # warm-up on the side stream
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            pkv.paged_decode_attention(*args, out=out, workspace=wsr, status=st)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(4):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pkv.check_status(st) == 0
    rows = np.random.default_rng(1).choice(w.batch * w.n_q_heads, 200, replace=False)
    compare_attention(ref, inp, "bf16", rows=np.sort(rows))


def test_decode_step_append_then_attend():
    """The token appended this step is attended to (seq_lens counts it)."""
    w = W.workload(2, batch=7, len_lo=1, len_hi=500)
    inp = W.make_decode_inputs(w, "cuda", with_logits=False)
    Kh, Vh = host(inp["k_cache"]), host(inp["v_cache"])
    pkv.kv_append(inp["k_new"], inp["v_new"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                  inp["seq_lens"])
    out = run_attention(inp)
    torch.cuda.synchronize()
    oracle.kv_append(host(inp["k_new"]), host(inp["v_new"]), Kh, Vh, host(inp["block_tables"]),
                     host(inp["seq_lens"]), w.block_size)
    ref, _, _ = oracle.paged_attention(host(inp["q"]), Kh, Vh, host(inp["block_tables"]), host(inp["seq_lens"]))
    got = out.float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= 2e-2 + 2e-2 * np.abs(ref))


# ----------------------------------------------------------------- sampler
@pytest.mark.parametrize("num,batch,vocab", [(1, None, None), (2, 16, None), (4, 64, None), (5, 64, 20000),
                                             (5, 32, None), (2, 8, 300001), (5, 24, 1001),
                                             (5, 6, 1 << 23)])  # the largest vocabulary the entry point takes
def test_sampler_parity(num, batch, vocab):
    w = W.workload(num)
    s = W.make_sampler_inputs(w, "cuda", batch=batch, vocab=vocab)
    st = pkv.new_status()
    tok = pkv.sample_tokens(*sampler_args(s), status=st)
    tok2 = pkv.sample_tokens(*sampler_args(s))
    torch.cuda.synchronize()
    assert pkv.check_status(st) == 0
    assert torch.equal(tok, tok2), "sampler is not deterministic"
    c = compare_tokens(tok, s)
    print(f"workload {num} B={c['rows']}: mismatches {c['mismatches']} (all exempt), "
          f"exempt draws {c['exempt_draw']}, exempt cuts {c['exempt_cut']}")


def test_sampler_special_rows():
    V = 4099
    g = torch.Generator().manual_seed(3)
    rows = []
    params = []

    def add(z, T=1.0, k=0, p=1.0, seed=7, off=0):
        rows.append(z)
        params.append((T, k, p, seed, off))
    base = torch.randn(V, generator=g)
    add(base.clone(), T=0.0)                                  # greedy
    zt = base.clone(); zt[[5, 900, 4000]] = 9.0
    add(zt, T=0.0)                                            # greedy tie -> lowest id (5)
    add(base.clone(), T=0.8, k=1)                             # k = 1 -> argmax
    add(base.clone(), T=0.8, p=1e-9)                          # p -> 0+ -> argmax
    add(base.clone(), T=1e-4)                                 # T -> 0+ -> argmax
    add(base.clone(), T=1.3, k=V + 10, p=0.7)                 # k beyond V -> off
    zb = base.clone(); zb[::3] = float("-inf")
    add(zb, T=0.9, k=40, p=0.9)                               # banned tokens
    zn = base.clone(); zn[17] = float("nan")
    add(zn)                                                   # NaN -> error, -1
    add(torch.full((V,), float("-inf")))                      # all banned -> error, -1
    add(base.clone(), T=-1.0)                                 # T < 0 -> error
    add(base.clone(), T=1.0, p=0.0)                           # p <= 0 -> error
    zi = base.clone(); zi[3] = float("inf")
    add(zi)                                                   # +inf -> error
    zz = torch.zeros(V); zz[1::2] = -0.0
    add(zz, T=1.0, k=7, p=0.5)                                # +-0 ties -> id order
    add((base * 40).clone(), T=0.5, k=1000, p=0.99)           # very peaked
    add(torch.full((V,), 3.0), T=1.0, k=10)                   # all equal, top-k by id
    add(torch.full((V,), 1.0), T=1.0, p=0.5, seed=11)         # all equal, top-p only (exact fallback)
    add(base.clone(), T=0.9, k=3000, p=0.9)                   # top-k beyond the gather list (fallback)
    add(base.clone(), T=0.6, p=0.3)                           # top-p only, narrow nucleus
    zs = base.clone(); zs[100] += 30.0
    add(zs, T=1.0, p=0.999999)                                # one dominant token, p near 1
    logits = torch.stack(rows).float().cuda()
    B = logits.shape[0]
    s = dict(logits=logits,
             temperature=torch.tensor([p[0] for p in params], dtype=torch.float32, device="cuda"),
             top_k=torch.tensor([p[1] for p in params], dtype=torch.int32, device="cuda"),
             top_p=torch.tensor([p[2] for p in params], dtype=torch.float32, device="cuda"),
             seeds=torch.tensor([p[3] for p in params], dtype=torch.int64, device="cuda"),
             offsets=torch.tensor([p[4] for p in params], dtype=torch.int64, device="cuda"))
    st = pkv.new_status()
    tok = pkv.sample_tokens(*sampler_args(s), status=st).cpu().numpy()
    code = pkv.check_status(st)
    assert code in (1, 6)
    am = int(torch.argmax(base))
    assert tok[0] == am and tok[1] == 5 and tok[2] == am and tok[3] == am and tok[4] == am
    assert tok[7] == -1 and tok[8] == -1 and tok[9] == -1 and tok[10] == -1 and tok[11] == -1
    assert tok[14] < 10
    assert tok[15] < V // 2 + 1                               # equal masses: the nucleus is the lowest ids
    c = compare_tokens(torch.from_numpy(tok), s)
    assert list(c["status"][7:12]) == [6, 6, 1, 1, 6]


def test_sampler_small_top_k_lists():
    """Top-k from 1 to 128 on the cluster kernel, with and without min-p: the
    candidate lists (every logit in the bins up to the one holding the k-th
    largest) take the rank-0 finish with eight threads per candidate up to 64
    candidates, four up to 128, and the sort beyond; plain and peaked rows,
    top-p on and off.  Every row matches the float64 oracle (exemptions as in
    the other sampler tests)."""
    from tests.gpu_helpers import EXEMPT
    rng = np.random.default_rng(71)
    B, V = 96, 50000
    z = (rng.standard_normal((B, V)) * rng.choice([0.5, 1.0, 2.0], (B, 1))).astype(np.float32)
    z[1::4, rng.integers(V)] += 10.0
    T = rng.uniform(0.4, 1.5, B).astype(np.float32)
    k = rng.choice([1, 2, 31, 32, 33, 63, 64, 65, 100, 127, 128], B).astype(np.int32)
    p = rng.choice([0.30011, 0.90007, 1.0], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    mp = np.where(rng.random(B) < 0.3, 0.02, 0.0).astype(np.float32)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    for with_min_p in (False, True):
        st = pkv.new_status()
        tok = pkv.sample_tokens(cu(z), cu(T), cu(k), cu(p), cu(seeds.view(np.int64)), cu(offs.view(np.int64)),
                                status=st, min_p=cu(mp) if with_min_p else None)
        got = tok.cpu().numpy()
        assert pkv.check_status(st) == 0
        exempt = 0
        for b in range(B):
            r = oracle.sample_row(z[b], float(T[b]), int(k[b]), float(p[b]), int(seeds[b]), int(offs[b]),
                                  min_p=float(mp[b]) if with_min_p else 0.0)
            if got[b] != r["token"]:
                assert r["draw_margin"] < EXEMPT or r["cut_margin"] < EXEMPT, (b, int(got[b]), r)
                exempt += 1
        assert exempt <= 2
