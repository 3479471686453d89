"""Host-side checks of the seeded input generators (CPU only)."""
import torch

from paged_kv_decode_table_gb300 import workloads as W


def _check_tables(w, inp):
    lens = inp["seq_lens"].tolist()
    bt = inp["block_tables"]
    nb = inp["num_blocks"]
    used = []
    for b, L in enumerate(lens):
        n = -(-L // w.block_size)
        row = bt[b].tolist()
        assert all(0 <= x < nb for x in row[:n])
        assert all(x == -1 for x in row[n:])
        used += row[:n]
    assert len(used) == len(set(used)), "a physical block is owned by two sequences"
    return used


def test_tiny_lab_workload():
    w = W.workload(1)
    inp = W.make_decode_inputs(w)
    assert inp["seq_lens"].tolist() == [9, 13]
    assert inp["num_blocks"] == 12
    used = _check_tables(w, inp)
    assert len(used) == 7                       # 3 + 4 blocks of 4 tokens
    assert inp["k_cache"].shape == (12, 2, 4, 4) and inp["k_cache"].dtype == torch.float32
    assert inp["logits"].shape == (2, 22)


def test_seeded_and_reproducible():
    w = W.workload(2, batch=6, len_hi=700)
    a = W.make_decode_inputs(w)
    b = W.make_decode_inputs(w)
    for k in ("seq_lens", "block_tables", "k_cache", "q", "logits"):
        assert torch.equal(a[k], b[k])
    assert a["k_cache"].dtype == torch.bfloat16


def test_fragmented_pool_has_holes():
    w = W.workload(4, batch=40)
    inp = W.make_decode_inputs(w, with_logits=False)
    used = _check_tables(w, inp)
    assert inp["num_blocks"] >= 1.25 * len(used) - 1
    assert 0 < len(used) < inp["num_blocks"]
    lens = inp["seq_lens"]
    assert int(lens.min()) >= 128 and int(lens.max()) <= 1024


def test_sampler_stress_inputs():
    w = W.workload(5)
    s = W.make_sampler_inputs(w, batch=16, vocab=1000)
    assert s["logits"].shape == (16, 1000)
    assert set(s["top_k"].tolist()) <= {0, 20, 50, 1000}
    assert set(round(x, 2) for x in s["top_p"].tolist()) <= {0.8, 0.95, 1.0}
    t = s["temperature"]
    assert float(t.min()) >= 0.5 and float(t.max()) <= 1.5
    # peaked half: the spike stands ~12 above the row
    peak = s["logits"][:8].max(dim=1).values
    assert float(peak.min()) > 8.0
    assert float(s["logits"][8:].abs().max()) < 1.0


def test_step_bytes_accounting():
    w = W.workload(2, batch=2)
    sl = torch.tensor([16, 33], dtype=torch.int32)
    by = W.step_bytes(w, sl)
    kv = (16 + 33) * 8 * 128 * 2 * 2
    assert W.kv_bytes(w, sl) == kv
    assert by["attention"] == kv + 2 * 2 * 32 * 128 * 2 + 4 * (1 + 3) + 4 * 2
