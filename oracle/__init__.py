"""CPU float64 oracle for the paged-KV decode step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The CUDA library in
``paged_kv_decode_table_gb300`` never imports, links or calls it, and the two
share no code: this package wraps ``pkv_oracle.c`` (plain C, float64, OpenMP)
through ctypes.

What each function follows (web pages cited by title and section):

* ``kv_append`` / ``gather``: "Bai Lab tong hop -- Inference Engineering",
  block [6] KV state manager (KVPool.write / KVPool.gather).
* ``paged_attention``: same lab, block [5] forward (two-pass softmax of
  q.K/sqrt(d) over every cached position, times V); GQA head grouping from
  "Suy luan & Toi uu hoa (Inference)" section 3.1.
* ``attention_split_row``: the online-softmax merge of "Suy luan & Toi uu hoa
  (Inference)" section 4.1, used only to pin the split algebra.
* ``sample_row`` / ``sample_batch``: temperature, top-k, top-p and the nucleus
  renormalisation of "Suy luan & Toi uu hoa (Inference)" section 1.2, with the
  tie rules of "LLM inference serving tutorial" section 3.1 and the filter order
  and draw order of the lab's block [8].
* ``philox4x64_10`` / ``uniform``: Salmon et al., SC'11.
* ``spec_verify_row`` / ``uniform_at``: speculative rejection sampling of
  "Suy luan & Toi uu hoa (Inference)" section 5.2 (accept with probability
  min(1, p/q), residual max(0, p - q) on rejection, a bonus token when all
  drafts are accepted), with the KV roll-back of "LLM inference serving
  tutorial" section 7 / Q16.
* ``process_logits``: hard constraint masks and the frequency / presence /
  sign-aware repetition penalties of "LLM inference serving tutorial" sections
  3.2-3.3, in the section 3.1 pipeline order; ``sample_row(min_p=...)`` adds
  min-p (section 3.1 and Q4) after top-p.
* ``kv_append_chunk`` / ``prefill_attention``: a prefill chunk of several
  tokens per sequence written through the block table and its causal attention
  over the cached prefix and the chunk ("Suy luan & Toi uu hoa (Inference)"
  2.1; "LLM inference serving tutorial" 5.4; the lab's prefill).
* ``copy_blocks``: the copy half of copy-on-write, "LLM inference serving
  tutorial" section 4.2.
* ``oracle.blocks`` (pure Python): reference-counted block sharing, fork,
  copy-on-write and idempotent reclaim ("LLM inference serving tutorial"
  sections 4.1, 4.2, 1.7 and appendix A [D07]-[D08]).

Parity status: every function above is pinned by ``tests/test_oracle_*.py``
(golden fixtures, closed forms, a library attention routine, brute force over
tiny vocabularies, numpy's Philox, and a chi-square draw test).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
INVALID_ARG = 1
DEVICE_BOUNDS = 4
NONFINITE = 6

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` with gcc (float64, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f32, f64, u64 = (ctypes.c_int, ctypes.c_longlong, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_uint64)
            lib.oracle_philox4x64_10.argtypes = [P, P, P]
            lib.oracle_philox4x64_10.restype = None
            lib.oracle_uniform.argtypes = [u64, u64]
            lib.oracle_uniform.restype = f64
            lib.oracle_kv_append.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32]
            lib.oracle_kv_append.restype = i32
            lib.oracle_gather.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, P]
            lib.oracle_gather.restype = i32
            lib.oracle_paged_attention.argtypes = [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32,
                                                   i32, i32, f64, P, i64, P]
            lib.oracle_paged_attention.restype = i32
            lib.oracle_attention_split_row.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                       i32, i32, i32, i32, f64, i32]
            lib.oracle_attention_split_row.restype = i32
            lib.oracle_sample_row.argtypes = [P, i32, f32, i32, f32, u64, u64, P, P, P, P, P]
            lib.oracle_sample_row.restype = i32
            lib.oracle_sample_batch.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P, P, P]
            lib.oracle_sample_batch.restype = i32
            lib.oracle_copy_blocks.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32]
            lib.oracle_copy_blocks.restype = i32
            lib.oracle_uniform_at.argtypes = [u64, u64, u64]
            lib.oracle_uniform_at.restype = f64
            lib.oracle_spec_verify_row.argtypes = [P, P, P, i32, i32, f32, u64, u64, i32, P, P, P, P, P]
            lib.oracle_spec_verify_row.restype = i32
            lib.oracle_sample_row_ex.argtypes = [P, i32, f32, i32, f32, f32, u64, u64, P, P, P, P, P]
            lib.oracle_sample_row_ex.restype = i32
            lib.oracle_sample_row_typical.argtypes = [P, i32, f32, f32, u64, u64, P, P, P, P, P, P, P]
            lib.oracle_sample_row_typical.restype = i32
            lib.oracle_process_logits.argtypes = [P, i32, i32, P, P, P, P, P, P, P]
            lib.oracle_process_logits.restype = i32
            lib.oracle_kv_append_chunk.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32]
            lib.oracle_kv_append_chunk.restype = i32
            lib.oracle_prefill_attention.argtypes = [P, P, P, P, i32, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                                     f64, P, i64, P]
            lib.oracle_prefill_attention.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError(f"oracle element type must be float32 or uint16 (bf16 bits), got {a.dtype}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def philox4x64_10(counter, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint64).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).reshape(2))
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, offset: int) -> float:
    return float(_load().oracle_uniform(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1)))


def kv_append(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, block_size) -> int:
    """In-place append of one token per sequence into numpy pools [NB, Hkv, BS, D]."""
    NB, Hkv, BS, D = k_cache.shape
    assert BS == block_size
    B = seq_lens.shape[0]
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    return int(_load().oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(bt), bt.shape[1], _ptr(sl), B, Hkv, D, BS, NB,
                                        _dtype_code(k_cache)))


def copy_blocks(k_cache, v_cache, src, dst) -> int:
    """In-place copy of whole physical blocks src[i] -> dst[i] in numpy pools [NB, Hkv, BS, D]."""
    NB, Hkv, BS, D = k_cache.shape
    s_ = np.ascontiguousarray(src, dtype=np.int32)
    d_ = np.ascontiguousarray(dst, dtype=np.int32)
    return int(_load().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(s_), _ptr(d_), s_.shape[0],
                                          Hkv, D, BS, NB, _dtype_code(k_cache)))


def uniform_at(seed: int, offset: int, j: int) -> float:
    """Uniform number j of the request stream (seed, offset); j = 0 is uniform()."""
    return float(_load().oracle_uniform_at(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), int(j)))


def spec_verify_row(target_logits, draft_logits, draft_tokens, temperature: float, seed: int, offset: int,
                    seq_len: int):
    """Speculative verification of one request.  target_logits [gamma+1, V],
    draft_logits [gamma, V] float32, draft_tokens [gamma] int32.  Returns dict
    (status, tokens [gamma+1], n_acc, seq_len_out, test_margin, draw_margin)."""
    zt = np.ascontiguousarray(target_logits, dtype=np.float32)
    g1, V = zt.shape
    gamma = g1 - 1
    zd = np.ascontiguousarray(draft_logits, dtype=np.float32).reshape(max(gamma, 0), V)
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(gamma)
    tok = np.zeros(gamma + 1, np.int32)
    n = ctypes.c_int32()
    so = ctypes.c_int32()
    tm, dm = ctypes.c_double(), ctypes.c_double()
    st = _load().oracle_spec_verify_row(_ptr(zt), _ptr(zd) if gamma else None, _ptr(x) if gamma else None, gamma,
                                        V, float(temperature), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                        int(seq_len), _ptr(tok), ctypes.byref(n), ctypes.byref(so),
                                        ctypes.byref(tm), ctypes.byref(dm))
    return dict(status=int(st), tokens=tok, n_acc=n.value, seq_len_out=so.value, test_margin=tm.value,
                draw_margin=dm.value)


def kv_append_chunk(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, q_start) -> int:
    """In-place append of n_b = q_start[b+1] - q_start[b] tokens per sequence (rows of the packed
    [T, Hkv, D] k_new / v_new) at positions seq_lens[b] - n_b .. seq_lens[b] - 1."""
    NB, Hkv, BS, D = k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    B = sl.shape[0]
    return int(_load().oracle_kv_append_chunk(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                              bt.shape[1], _ptr(sl), _ptr(qs), B, Hkv, D, BS, NB,
                                              _dtype_code(k_cache)))


def prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, q_start, scale: float = 0.0, rows=None):
    """Causal chunk attention; q [T, Hq, D].  Returns (out float64 [n, D], status, max |sum w - 1|)."""
    T, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    assert D == D2
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    B = sl.shape[0]
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n = T * Hq if r is None else r.shape[0]
    out = np.zeros((n, D), dtype=np.float64)
    werr = ctypes.c_double(0.0)
    st = _load().oracle_prefill_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _dtype_code(q), _ptr(bt),
                                          bt.shape[1], _ptr(sl), _ptr(qs), B, Hq, Hkv, D, BS, NB, float(scale),
                                          None if r is None else _ptr(r), n, ctypes.byref(werr))
    return out, int(st), float(werr.value)


def gather(cache, block_tables, b: int, L: int, h: int) -> np.ndarray:
    """Contiguous float64 [L, D] copy of sequence b, KV head h."""
    NB, Hkv, BS, D = cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    out = np.zeros((L, D), dtype=np.float64)
    st = _load().oracle_gather(_ptr(cache), _ptr(bt), bt.shape[1], b, L, h, Hkv, D, BS, NB,
                               _dtype_code(cache), _ptr(out))
    if st != OK:
        raise ValueError(f"gather: status {st}")
    return out


def paged_attention(q, k_cache, v_cache, block_tables, seq_lens, scale: float = 0.0, rows=None):
    """float64 attention output: [B, Hq, D] (rows=None) or [len(rows), D] for flat rows b*Hq+qh.

    Returns (out, status, max |sum(weights) - 1|)."""
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    assert D == D2
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if rows is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        rptr, nrows = None, 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((rows.shape[0], D), dtype=np.float64)
        rptr, nrows = _ptr(rows), rows.shape[0]
    werr = ctypes.c_double(0.0)
    st = _load().oracle_paged_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _dtype_code(q), _ptr(bt), bt.shape[1], _ptr(sl), B, Hq,
                                        Hkv, D, BS, NB, float(scale), rptr, nrows,
                                        ctypes.byref(werr))
    return out, int(st), float(werr.value)


def attention_split_row(q, k_cache, v_cache, block_tables, seq_lens, b: int, qh: int,
                        chunk_tokens: int, scale: float = 0.0) -> np.ndarray:
    B, Hq, D = q.shape
    NB, Hkv, BS, _ = k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    out = np.zeros(D, dtype=np.float64)
    st = _load().oracle_attention_split_row(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _dtype_code(q), _ptr(bt), bt.shape[1], b, qh,
                                            int(seq_lens[b]), Hq, Hkv, D, BS, NB, float(scale),
                                            int(chunk_tokens))
    if st != OK:
        raise ValueError(f"split row: status {st}")
    return out


def sample_row(z, temperature: float, top_k: int, top_p: float, seed: int, offset: int,
               want_probs: bool = False, min_p: float = 0.0):
    """One row (min_p > 0: min-p after top-p). Returns dict(token, status,
    draw_margin, cut_margin, n_kept[, probs])."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    V = z.shape[0]
    tok = ctypes.c_int32(0)
    dm = ctypes.c_double(0)
    cm = ctypes.c_double(0)
    nk = ctypes.c_int32(0)
    probs = np.zeros(V, dtype=np.float64) if want_probs else None
    st = _load().oracle_sample_row_ex(_ptr(z), V, float(temperature), int(top_k), float(top_p), float(min_p),
                                   int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                   ctypes.byref(tok), ctypes.byref(dm), ctypes.byref(cm),
                                   ctypes.byref(nk), _ptr(probs) if want_probs else None)
    res = dict(token=int(tok.value), status=int(st), draw_margin=float(dm.value),
               cut_margin=float(cm.value), n_kept=int(nk.value))
    if want_probs:
        res["probs"] = probs
    return res


def sample_row_typical(z, temperature: float, typical_p: float, seed: int, offset: int, want_probs: bool = False):
    """One row of typical sampling. Returns dict(token, status, draw_margin,
    cut_margin, order_margin, entropy, n_kept[, probs])."""
    z = np.ascontiguousarray(z, dtype=np.float32)
    V = z.shape[0]
    tok = ctypes.c_int32(0)
    dm, cm, ctm, ent = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    nk = ctypes.c_int32(0)
    probs = np.zeros(V, dtype=np.float64) if want_probs else None
    st = _load().oracle_sample_row_typical(_ptr(z), V, float(temperature), float(typical_p),
                                        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), ctypes.byref(tok),
                                        ctypes.byref(dm), ctypes.byref(cm), ctypes.byref(ctm), ctypes.byref(ent),
                                        ctypes.byref(nk), _ptr(probs) if want_probs else None)
    res = dict(token=int(tok.value), status=int(st), draw_margin=float(dm.value), cut_margin=float(cm.value),
               order_margin=float(ctm.value), entropy=float(ent.value), n_kept=int(nk.value))
    if want_probs:
        res["probs"] = probs
    return res


def process_logits(logits, mask=None, row_ptr=None, tokens=None, counts=None, rep=None, freq=None, pres=None):
    """Masks and penalties in place on float32 logits [B, V]; returns the status."""
    B, V = logits.shape
    arr = lambda a, t: None if a is None else np.ascontiguousarray(a, dtype=t)
    m, rp, tk, ct = arr(mask, np.uint32), arr(row_ptr, np.int32), arr(tokens, np.int32), arr(counts, np.int32)
    r, f, p = arr(rep, np.float32), arr(freq, np.float32), arr(pres, np.float32)
    P = lambda a: None if a is None else _ptr(a)
    return int(_load().oracle_process_logits(_ptr(logits), B, V, P(m), P(rp), P(tk), P(ct), P(r), P(f), P(p)))


def sample_batch(logits, temperature, top_k, top_p, seeds, offsets):
    """All rows. Returns dict of arrays: tokens, status, draw_margin, cut_margin, n_kept."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    B, V = logits.shape
    t = np.ascontiguousarray(temperature, dtype=np.float32)
    k = np.ascontiguousarray(top_k, dtype=np.int32)
    p = np.ascontiguousarray(top_p, dtype=np.float32)
    s = np.ascontiguousarray(np.asarray(seeds).astype(np.uint64))
    o = np.ascontiguousarray(np.asarray(offsets).astype(np.uint64))
    tokens = np.zeros(B, dtype=np.int32)
    dm = np.zeros(B, dtype=np.float64)
    cm = np.zeros(B, dtype=np.float64)
    nk = np.zeros(B, dtype=np.int32)
    st = np.zeros(B, dtype=np.int32)
    _load().oracle_sample_batch(_ptr(logits), B, V, _ptr(t), _ptr(k), _ptr(p), _ptr(s), _ptr(o),
                                _ptr(tokens), _ptr(dm), _ptr(cm), _ptr(nk), _ptr(st))
    return dict(tokens=tokens, status=st, draw_margin=dm, cut_margin=cm, n_kept=nk)
