"""The library's reference-counted block pool (pkv_block_pool_*, pkv_seq_*)
against the plain oracle model (oracle.blocks), on CPU.

Both sides run the same seeded sequence of add / fork / append / free calls.
Block ids are each side's own policy, so what is compared is what the method
fixes: the status of every call, whether a copy-on-write pair was produced,
every sequence's length, the number of free blocks, and the sharing structure
(which logical blocks of which sequences name the same physical block), with
physical ids relabelled in order of first appearance.  Also the [D08] case
through the library, reclaim idempotence and atomic failure.
"""
import random

import pytest

import paged_kv_decode_table_gb300 as pkv
from oracle import blocks as OB

CODE = {"ok": 0, "invalid": 1, "capacity": 7}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_decode_table_gb300 import build
    build.build()
    pkv.load_library()


def _structure(tables: dict):
    label, out = {}, {}
    for s in sorted(tables, key=str):
        row = []
        for b in tables[s]:
            if b not in label:
                label[b] = len(label)
            row.append(label[b])
        out[s] = row
    return out


def _lib_tables(pool, seqs):
    if not seqs:
        return {}
    bt, sl = pool.tables(seqs)
    res = {}
    for i, s in enumerate(seqs):
        n = -(-int(sl[i]) // pool.block_size)
        row = bt[i].tolist()
        assert all(x == -1 for x in row[n:])
        res[s] = row[:n]
    return res


def _call(fn, *a):
    try:
        r = fn(*a)
        return 0, r
    except pkv.PkvError as e:
        return e.code, None


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_oracle(seed):
    rng = random.Random(seed)
    NB, BS, MB = 24, 4, 6
    pool = pkv.BlockPool(NB, BS, MB)
    ref = OB.OracleBlockManager(NB, BS, MB)
    live, next_id = [], 0
    for step in range(300):
        op = rng.choices(["add", "fork", "append", "free"], weights=[2, 2, 8, 2])[0]
        if op == "add" or not live:
            length = rng.randint(0, 14)
            a = ref.add(next_id, length)
            b, _ = _call(pool.add, next_id, length)
            assert b == CODE[a], (step, op)
            if a == "ok":
                live.append(next_id)
            next_id += 1
        elif op == "fork":
            parent = rng.choice(live)
            a = ref.fork(parent, next_id)
            b, _ = _call(pool.fork, parent, next_id)
            assert b == CODE[a], (step, op)
            if a == "ok":
                live.append(next_id)
            next_id += 1
        elif op == "append":
            s = rng.choice(live)
            a, pair_ref = ref.append(s)
            b, pair_lib = _call(pool.append, s)
            assert b == CODE[a], (step, op)
            assert (pair_ref is None) == (pair_lib is None), (step, op)
            if pair_lib is not None:
                # the copy's source is the block the sequence named before
                assert pool.refcount(pair_lib[1]) == 1 and pool.refcount(pair_lib[0]) >= 1
        else:
            s = rng.choice(live + [10_000])   # sometimes an unknown / reclaimed id
            a = ref.free(s)
            b, _ = _call(pool.free, s)
            assert b == CODE[a] == 0
            if s in live:
                live.remove(s)
        ref.check()
        assert pool.num_free() == len(ref.free_blocks())
        for s in live:
            assert pool.length(s) == ref.lengths[s]
        assert _structure(_lib_tables(pool, live)) == _structure({s: ref.tables[s] for s in live})
    for s in list(live):
        pool.free(s)
        pool.free(s)
    assert pool.num_free() == NB
    assert all(pool.refcount(b) == 0 for b in range(NB))


def test_d08_through_the_library():
    pool = pkv.BlockPool(16, 4, 8)
    pool.add(1, 4)
    pool.fork(1, 2)
    assert [pool.append(1) for _ in range(2)] == [None, None]
    assert [pool.append(2) for _ in range(3)] == [None, None, None]
    assert 16 - pool.num_free() == 3
    bt, sl = pool.tables([1, 2])
    assert sl.tolist() == [6, 7] and bt[0, 0] == bt[1, 0] and bt[0, 1] != bt[1, 1]
    assert pool.refcount(int(bt[0, 0])) == 2


def test_copy_on_write_pair_and_refcounts():
    pool = pkv.BlockPool(8, 4, 4)
    pool.add(0, 6)
    pool.fork(0, 1)
    bt, _ = pool.tables([0])
    tail = int(bt[0, 1])
    pair = pool.append(1)
    assert pair is not None and pair[0] == tail
    bt2, sl2 = pool.tables([0, 1])
    assert int(bt2[1, 1]) == pair[1] and int(bt2[0, 1]) == tail and sl2.tolist() == [6, 7]
    assert pool.refcount(tail) == 1 and pool.refcount(pair[1]) == 1
    assert pool.append(0) is None


def test_failures_change_nothing():
    pool = pkv.BlockPool(3, 4, 8)
    pool.add(0, 8)
    with pytest.raises(pkv.PkvError) as e:
        pool.add(1, 8)
    assert e.value.code == 7
    with pytest.raises(pkv.PkvError):
        pool.add(0, 1)          # duplicate id
    with pytest.raises(pkv.PkvError):
        pool.fork(5, 6)         # unknown parent
    assert pool.num_free() == 1 and pool.length(0) == 8 and pool.length(1) == -1
    pool.add(2, 4)
    with pytest.raises(pkv.PkvError) as e:
        pool.append(0)          # position 8 opens a block; none is free
    assert e.value.code == 7 and pool.length(0) == 8
    pool.free(0)
    pool.free(0)
    assert pool.num_free() == 2
