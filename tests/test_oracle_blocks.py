"""Pins of the block-sharing oracle (oracle.blocks, oracle.copy_blocks).

The worked numbers are those of "LLM inference serving tutorial", appendix A
[D07]-[D08] (stored in tests/golden/kv_block_sharing_d07_d08.txt with their
citation); the rest are invariants the tutorial states in sections 4.2 and 1.7:
reference counts equal the number of tables naming a block, a shared partial
tail block is copied before it is written, and reclaiming twice frees nothing
twice.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import blocks as OB

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_block_sharing_d07_d08.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split("=", 1)
            vals[k.strip()] = [int(x) for x in v.split(",")]
    return vals


def test_d07_bytes_and_slots():
    g = _golden()
    m = OB.kv_bytes_per_token(2, 2, 4, 2)
    assert m == g["m_token"][0]
    logical, allocated = OB.block_alloc_slots([1, 5], block_size=4)
    assert [logical, allocated] == g["slots_logical_allocated"]
    assert [logical * m, allocated * m] == g["bytes_logical_allocated"]


def test_d08_sharing_one_full_block_saves_one():
    g = _golden()
    assert OB.physical_blocks_no_sharing([6, 7], 4) == g["physical_no_sharing"][0]
    mgr = OB.OracleBlockManager(16, 4, 8)
    assert mgr.add("a", 4) == "ok"           # the shared, full prefix block
    assert mgr.fork("a", "b") == "ok"
    for _ in range(2):
        assert mgr.append("a") == ("ok", None)
    for _ in range(3):
        assert mgr.append("b") == ("ok", None)  # full shared block: no copy needed
    assert (mgr.lengths["a"], mgr.lengths["b"]) == (6, 7)
    mgr.check()
    used = sum(1 for r in mgr.ref if r > 0)
    assert used == g["physical_with_sharing"][0]


def test_shared_partial_tail_is_copied_before_write():
    mgr = OB.OracleBlockManager(8, 4, 4)
    assert mgr.add(0, 6) == "ok"       # blocks [x, y], y holds 2 tokens
    tail = mgr.tables[0][1]
    assert mgr.fork(0, 1) == "ok"
    assert mgr.ref[tail] == 2
    st, pair = mgr.append(1)
    assert st == "ok" and pair is not None and pair[0] == tail
    assert mgr.tables[1][1] == pair[1] != tail and mgr.tables[0][1] == tail
    assert mgr.ref[tail] == 1 and mgr.ref[pair[1]] == 1
    # the other sharer now owns the tail alone: no copy on its next write
    assert mgr.append(0) == ("ok", None)
    mgr.check()


def test_reclaim_is_idempotent_and_returns_every_block():
    mgr = OB.OracleBlockManager(10, 4, 4)
    mgr.add("p", 9)
    for c in range(3):
        mgr.fork("p", c)
    for c in range(3):
        mgr.append(c)
    mgr.check()
    for s in ["p", 0, 1, 2]:
        assert mgr.free(s) == "ok"
        assert mgr.free(s) == "ok"     # second reclaim changes nothing
        mgr.check()
    assert len(mgr.free_blocks()) == 10 and all(r == 0 for r in mgr.ref)


def test_capacity_failure_changes_nothing():
    mgr = OB.OracleBlockManager(3, 4, 8)
    assert mgr.add(0, 8) == "ok"
    before = (list(mgr.ref), {k: list(v) for k, v in mgr.tables.items()})
    assert mgr.add(1, 8) == "capacity"
    assert (list(mgr.ref), {k: list(v) for k, v in mgr.tables.items()}) == before
    assert mgr.add(2, 40) == "invalid"   # beyond max_blocks_per_seq * block_size


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_copy_blocks_moves_whole_blocks(dtype):
    rng = np.random.default_rng(7)
    NB, Hkv, BS, D = 9, 2, 4, 8
    if dtype == np.float32:
        K = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float32)
        V = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float32)
    else:
        K = rng.integers(0, 1 << 16, (NB, Hkv, BS, D), dtype=np.uint16)
        V = rng.integers(0, 1 << 16, (NB, Hkv, BS, D), dtype=np.uint16)
    K0, V0 = K.copy(), V.copy()
    src, dst = np.array([1, 4, 6], np.int32), np.array([3, 0, 8], np.int32)
    assert oracle.copy_blocks(K, V, src, dst) == oracle.OK
    for s, d in zip(src, dst):
        np.testing.assert_array_equal(K[d], K0[s])
        np.testing.assert_array_equal(V[d], V0[s])
    untouched = [b for b in range(NB) if b not in set(dst.tolist())]
    np.testing.assert_array_equal(K[untouched], K0[untouched])
    np.testing.assert_array_equal(V[untouched], V0[untouched])
    # out-of-range ids are skipped and reported
    assert oracle.copy_blocks(K, V, np.array([1, 99], np.int32), np.array([2, 5], np.int32)) == oracle.DEVICE_BOUNDS
    np.testing.assert_array_equal(K[2], K0[1])
    np.testing.assert_array_equal(K[5], K0[5])


def test_copy_then_remap_gathers_the_same_sequence():
    """A sequence read through its old (shared) table equals the same sequence
    read through the remapped table after its tail block was copied."""
    rng = np.random.default_rng(3)
    NB, Hkv, BS, D = 8, 2, 4, 4
    K = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float32)
    V = rng.standard_normal((NB, Hkv, BS, D)).astype(np.float32)
    table = np.array([[5, 2, -1]], np.int32)
    L = 7
    before = [oracle.gather(K, table, 0, L, h) for h in range(Hkv)]
    oracle.copy_blocks(K, V, np.array([2], np.int32), np.array([6], np.int32))
    remapped = np.array([[5, 6, -1]], np.int32)
    for h in range(Hkv):
        np.testing.assert_array_equal(oracle.gather(K, remapped, 0, L, h), before[h])
