"""Plain model of reference-counted KV block sharing -- TEST INFRASTRUCTURE ONLY.

Follows "LLM inference serving tutorial" (wanshuiyin.github.io, ARIS-in-AI-Offer):

* section 4.1: the ideal KV payload per token is 2 * N_layer * N_kv_head *
  d_head * b bytes (K and V, b bytes per element);
* section 4.2: a block table maps each sequence's logical blocks to physical
  blocks; physical blocks are shared by reference count between common
  prefixes and beam branches; a shared, still-writable tail block is copied
  before it diverges (copy-on-write) instead of being written in place;
* section 1.7: reclaim decrements reference counts, a block returns to the
  allocator only when its last holder releases it, and reclaiming the same
  request twice must neither free a block twice nor leak one;
* appendix A [D07]-[D08]: logical vs allocated slots (lengths [1, 5] at block
  size 4 occupy 6 logical and 12 allocated slots), and two sequences of lengths
  6 and 7 that share one full block need 3 physical blocks instead of 4.

Everything is kept as plain Python lists and dicts; the block ids it hands out
are the lowest free ids, a policy of its own (the library's may differ; tests
compare the sharing structure, not the ids).
"""
from __future__ import annotations


def kv_bytes_per_token(n_layer: int, n_kv_head: int, d_head: int, bytes_per_elem: int) -> int:
    """Ideal KV payload of one token (section 4.1)."""
    return 2 * n_layer * n_kv_head * d_head * bytes_per_elem


def blocks_needed(length: int, block_size: int) -> int:
    return -(-length // block_size)


def block_alloc_slots(lengths, block_size: int):
    """(logical slots, allocated slots) of sequences that share nothing ([D07])."""
    logical = sum(lengths)
    allocated = sum(blocks_needed(n, block_size) * block_size for n in lengths)
    return logical, allocated


def physical_blocks_no_sharing(lengths, block_size: int) -> int:
    return sum(blocks_needed(n, block_size) for n in lengths)


class OracleBlockManager:
    """Reference-counted physical blocks; one table (list of block ids) per sequence."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.max_blocks_per_seq = max_blocks_per_seq
        self.ref = [0] * num_blocks
        self.tables = {}   # seq -> list of physical block ids
        self.lengths = {}  # seq -> tokens

    # -- helpers
    def free_blocks(self):
        return [b for b in range(self.num_blocks) if self.ref[b] == 0]

    def _new_block(self):
        free = self.free_blocks()
        if not free:
            return None
        b = free[0]
        self.ref[b] = 1
        return b

    # -- operations (each returns a status string; "ok" or the reason nothing changed)
    def add(self, seq, length):
        if seq in self.tables or length < 0:
            return "invalid"
        need = blocks_needed(length, self.block_size)
        if need > self.max_blocks_per_seq:
            return "invalid"
        if need > len(self.free_blocks()):
            return "capacity"
        self.tables[seq] = [self._new_block() for _ in range(need)]
        self.lengths[seq] = length
        return "ok"

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables:
            return "invalid"
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.ref[b] += 1
        return "ok"

    def append(self, seq):
        """Make room for one token; returns (status, copy pair or None)."""
        if seq not in self.tables:
            return "invalid", None
        table, pos = self.tables[seq], self.lengths[seq]
        pair = None
        if pos % self.block_size == 0:
            if len(table) >= self.max_blocks_per_seq:
                return "invalid", None
            b = self._new_block()
            if b is None:
                return "capacity", None
            table.append(b)
        else:
            tail = table[-1]
            if self.ref[tail] > 1:
                b = self._new_block()
                if b is None:
                    return "capacity", None
                self.ref[tail] -= 1
                table[-1] = b
                pair = (tail, b)
        self.lengths[seq] = pos + 1
        return "ok", pair

    def free(self, seq):
        if seq not in self.tables:
            return "ok"  # reclaiming twice is harmless
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
        del self.lengths[seq]
        return "ok"

    # -- invariants
    def check(self):
        """Reference counts equal the number of table entries naming each block."""
        count = [0] * self.num_blocks
        for t in self.tables.values():
            for b in t:
                count[b] += 1
        assert count == self.ref, "reference counts disagree with the tables"
        assert all(r >= 0 for r in self.ref)
        for s, t in self.tables.items():
            assert len(t) == blocks_needed(self.lengths[s], self.block_size)
