"""GPU parity of the cluster sampler when it runs one CTA per row with more
rows than SMs (vocabularies above the per-row kernel's 65536): the CTAs take
the rows heaviest first (top-p alone, then large top-k or no truncation, then
greedy, small top-k and invalid rows), so the row a CTA serves is computed on
the device.  Every row is compared with the float64 oracle (the same token
unless the oracle's draw or top-p cut lies within 1e-6 of an edge, counted, at
most max(1, B // 50)); invalid rows return -1 with their error code; the
tokens are identical to those of the same rows in a batch small enough to keep
its natural order.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_table_gb300 as pkv
from gpu_helpers import EXEMPT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _cu(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _sample(z, T, k, p, seeds, offs):
    st = pkv.new_status()
    tok = pkv.sample_tokens(_cu(z), _cu(T), _cu(k), _cu(p), _cu(seeds.view(np.int64)), _cu(offs.view(np.int64)),
                            status=st)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), pkv.check_status(st)


def _mixed(rng, B, V):
    z = (rng.standard_normal((B, V)) * rng.choice([0.1, 1.0, 2.0], (B, 1))).astype(np.float32)
    z[0::3, rng.integers(V)] += 12.0
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[::11] = 0.0
    k = rng.choice([0, 0, 20, 50, 300, 1000], B).astype(np.int32)
    p = rng.choice([0.80007, 0.95003, 1.0], B).astype(np.float32)
    seeds = rng.integers(0, 2**63, B).astype(np.uint64)
    offs = rng.integers(0, 1000, B).astype(np.uint64)
    return z, T, k, p, seeds, offs


@pytest.mark.parametrize("extra_rows", [48, 248])
def test_heaviest_first_rows_match_oracle(extra_rows):
    """#SM + 48 rows (one wave, some SMs with two rows) and #SM + 248 rows
    (two waves), V = 70000, every row class mixed, four invalid rows."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, V = sms + extra_rows, 70000
    rng = np.random.default_rng(40 + extra_rows)
    z, T, k, p, seeds, offs = _mixed(rng, B, V)
    bad = {5: "nan", 9: "neg_t", 17: "p0", 23: "all_inf"}
    z[5, 100] = np.nan
    T[9] = -1.0
    T[17], p[17] = 0.9, 0.0
    z[23] = -np.inf
    got, st = _sample(z, T, k, p, seeds, offs)
    assert st in (1, 6)
    assert all(got[b] == -1 for b in bad)
    exempt = 0
    for b in range(B):
        if b in bad:
            continue
        r = oracle.sample_row(z[b], float(T[b]), int(k[b]), float(p[b]), int(seeds[b]), int(offs[b]))
        assert r["status"] == 0
        if got[b] != r["token"]:
            assert r["draw_margin"] < EXEMPT or r["cut_margin"] < EXEMPT, (b, int(got[b]), r)
            exempt += 1
    assert exempt <= max(1, B // 50)
    # the same rows, a few at a time (one row per SM at most: the natural order)
    for lo in range(0, B, 64):
        sl = slice(lo, min(B, lo + 64))
        part, _ = _sample(z[sl], T[sl], k[sl], p[sl], seeds[sl], offs[sl])
        assert np.array_equal(part, got[sl]), lo
