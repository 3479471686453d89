"""Paged-KV decode step for GB300 (sm_103a).

Thin ctypes binding over the C ABI in ``include/pkv.h`` (``libpkv.so``, built
in-tree by ``paged_kv_decode_table_gb300.build``).  Every function here only
checks and marshals torch tensors (device, dtype, contiguity, shapes) and passes
raw device pointers plus the current CUDA stream; all arithmetic runs in the
library's CUDA kernels.  There is no CPU fallback: if the library cannot be
loaded, every call raises.

Calls (names follow the C ABI):
  kv_append(k_new, v_new, k_cache, v_cache, block_tables, seq_lens)
  paged_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, out=None, scale=0.0)
  sample_tokens(logits, temperature, top_k, top_p, seeds, offsets, tokens=None)
  copy_blocks(k_cache, v_cache, src, dst)
  spec_verify(target_logits, draft_logits, draft_tokens, seq_lens, temperature, seeds, offsets)
  apply_logits_processors(logits, allow_mask=None, row_ptr=None, tokens=None, counts=None, ...)
  kv_append_chunk(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, q_start)
  paged_prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, q_start, out=None, scale=0.0)
  BlockPool(num_blocks, block_size, max_blocks_per_seq)   host-side refcounted block ids
  DecodeStep(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, logits, ...).run()
      a whole decode step (append + attention + sampler) bound to fixed buffers
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["PkvError", "load_library", "library_path", "kv_append", "paged_decode_attention",
           "paged_decode_attention_append",
           "decode_workspace_bytes", "sample_tokens", "sample_workspace_bytes", "status_string",
           "new_status", "check_status", "STATUS", "copy_blocks", "BlockPool", "spec_verify",
           "spec_verify_workspace_bytes", "apply_logits_processors", "kv_append_chunk",
           "paged_prefill_attention", "DecodeStep", "test_set_wait_limit"]

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_CUDA",
          4: "PKV_ERR_DEVICE_BOUNDS", 5: "PKV_ERR_TIMEOUT", 6: "PKV_ERR_NONFINITE", 7: "PKV_ERR_CAPACITY"}
PKV_F32, PKV_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lib = None
_lock = threading.Lock()
_ws_cache: dict = {}


class PkvError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call} failed: {STATUS.get(code, code)} ({code})")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: run paged_kv_decode_table_gb300.build.build() first")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pkv_status_string.argtypes = [i32]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = i32
        lib.pkv_kv_append.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, P, P]
        lib.pkv_kv_append.restype = i32
        lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.pkv_decode_workspace_bytes.restype = sz
        lib.pkv_paged_decode_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, f32,
                                                   i32, P, sz, P, P]
        lib.pkv_paged_decode_attention.restype = i32
        lib.pkv_paged_decode_attention_append.argtypes = [P, P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                          i32, f32, i32, P, sz, P, P]
        lib.pkv_paged_decode_attention_append.restype = i32
        lib.pkv_sample_workspace_bytes.argtypes = [i32, i32]
        lib.pkv_sample_workspace_bytes.restype = sz
        lib.pkv_sample_tokens.argtypes = [P, P, i32, i32, P, P, P, P, P, P, sz, P, P]
        lib.pkv_sample_tokens.restype = i32
        i64 = ctypes.c_int64
        lib.pkv_kv_append_chunk.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, P, P]
        lib.pkv_kv_append_chunk.restype = i32
        lib.pkv_paged_prefill_attention.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                    f32, i32, P, P]
        lib.pkv_paged_prefill_attention.restype = i32
        lib.pkv_sample_tokens_ex.argtypes = [P, P, i32, i32, P, P, P, P, P, P, P, P]
        lib.pkv_sample_tokens_ex.restype = i32
        lib.pkv_sample_tokens_typical.argtypes = [P, P, i32, i32, P, P, P, P, P, P]
        lib.pkv_sample_tokens_typical.restype = i32
        lib.pkv_apply_logits_processors.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P, P]
        lib.pkv_apply_logits_processors.restype = i32
        lib.pkv_spec_verify_workspace_bytes.argtypes = [i32, i32]
        lib.pkv_spec_verify_workspace_bytes.restype = sz
        lib.pkv_spec_verify.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, P, P, P, P, sz, P, P]
        lib.pkv_spec_verify.restype = i32
        lib.pkv_copy_blocks.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P]
        lib.pkv_copy_blocks.restype = i32
        lib.pkv_block_pool_create.argtypes = [i32, i32, i32]
        lib.pkv_block_pool_create.restype = P
        lib.pkv_block_pool_destroy.argtypes = [P]
        lib.pkv_block_pool_destroy.restype = None
        lib.pkv_block_pool_num_free.argtypes = [P]
        lib.pkv_block_pool_num_free.restype = i32
        lib.pkv_block_pool_refcount.argtypes = [P, i32]
        lib.pkv_block_pool_refcount.restype = i32
        lib.pkv_seq_add.argtypes = [P, i64, i32]
        lib.pkv_seq_add.restype = i32
        lib.pkv_seq_fork.argtypes = [P, i64, i64]
        lib.pkv_seq_fork.restype = i32
        lib.pkv_seq_append.argtypes = [P, i64, P, P, P]
        lib.pkv_seq_append.restype = i32
        lib.pkv_seq_free.argtypes = [P, i64]
        lib.pkv_seq_free.restype = i32
        lib.pkv_seq_length.argtypes = [P, i64]
        lib.pkv_seq_length.restype = i32
        lib.pkv_block_tables.argtypes = [P, P, i32, P, P]
        lib.pkv_block_tables.restype = i32
        lib.pkv_test_set_wait_limit.argtypes = [ctypes.c_uint32, i32]
        lib.pkv_test_set_wait_limit.restype = i32
        _lib = lib
        return lib


def test_set_wait_limit(polls: int = 0, silent_cta: int = -1) -> None:
    """Failure-path test hook (pkv_test_set_wait_limit): the poll budget of the
    attention kernel's waits (0: the default) and one CTA whose loader issues
    no copy (-1: none).  Call with no arguments to restore the defaults."""
    _raise("pkv_test_set_wait_limit", load_library().pkv_test_set_wait_limit(int(polls), int(silent_cta)))


def status_string(code: int) -> str:
    return load_library().pkv_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_cuda(name: str, t: torch.Tensor, dtype=None, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PKV_F32
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"unsupported element type {t.dtype} (float32 or bfloat16)")


def _raise(name, code):
    if code != 0:
        raise PkvError(name, code)


def new_status(device="cuda") -> torch.Tensor:
    """A zeroed device status word to pass as `status=`."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor) -> int:
    """Read a device status word (synchronises); returns the code."""
    return int(status.item())


def kv_append(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, status=None):
    """Write k_new/v_new [B, Hkv, D] at position seq_lens[b]-1 of each sequence."""
    NB, Hkv, BS, D = k_cache.shape
    B = seq_lens.shape[0]
    dev = k_cache.device
    _check_cuda("k_cache", k_cache)
    _check_cuda("v_cache", v_cache, k_cache.dtype, k_cache.shape, dev)
    _check_cuda("k_new", k_new, k_cache.dtype, (B, Hkv, D), dev)
    _check_cuda("v_new", v_new, k_cache.dtype, (B, Hkv, D), dev)
    _check_cuda("block_tables", block_tables, torch.int32, device=dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [B, max_blocks_per_seq]")
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B,
                                        Hkv, D, BS, NB, _dtype_code(k_cache), _ptr(status),
                                        _stream(dev))
    _raise("pkv_kv_append", code)


def decode_workspace_bytes(B: int, Hq: int, D: int, num_sms: int = 0) -> int:
    return int(load_library().pkv_decode_workspace_bytes(B, Hq, D, num_sms))


def _workspace(dev, nbytes: int) -> torch.Tensor:
    key = (dev, nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
        _ws_cache.clear()
        _ws_cache[key] = ws
    return ws


def paged_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, out=None, scale: float = 0.0,
                           workspace=None, status=None):
    """GQA decode attention over the paged cache; returns out [B, Hq, D]."""
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    dev = q.device
    if D2 != D:
        raise ValueError("head_dim of q and the cache differ")
    _check_cuda("q", q)
    _check_cuda("k_cache", k_cache, q.dtype, device=dev)
    _check_cuda("v_cache", v_cache, q.dtype, k_cache.shape, dev)
    _check_cuda("block_tables", block_tables, torch.int32, device=dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [B, max_blocks_per_seq]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda("out", out, q.dtype, q.shape, dev)
    lib = load_library()
    need = int(lib.pkv_decode_workspace_bytes(B, Hq, D, 0))
    if workspace is None:
        with torch.cuda.device(dev):
            workspace = _workspace(dev, need)
    _check_cuda("workspace", workspace, device=dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = lib.pkv_paged_decode_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                          B, Hq, Hkv, D, BS, NB, float(scale), _dtype_code(q),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _ptr(status), _stream(dev))
    _raise("pkv_paged_decode_attention", code)
    return out


def paged_decode_attention_append(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, out=None,
                                  scale: float = 0.0, workspace=None, status=None):
    """kv_append(k_new, v_new, ...) then paged_decode_attention(q, ...) in one call; returns out."""
    B, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    dev = q.device
    if D2 != D:
        raise ValueError("head_dim of q and the cache differ")
    _check_cuda("q", q)
    _check_cuda("k_cache", k_cache, q.dtype, device=dev)
    _check_cuda("v_cache", v_cache, q.dtype, k_cache.shape, dev)
    _check_cuda("k_new", k_new, q.dtype, (B, Hkv, D), dev)
    _check_cuda("v_new", v_new, q.dtype, (B, Hkv, D), dev)
    _check_cuda("block_tables", block_tables, torch.int32, device=dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    if block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("block_tables must be [B, max_blocks_per_seq]")
    if out is None:
        out = torch.empty_like(q)
    _check_cuda("out", out, q.dtype, q.shape, dev)
    lib = load_library()
    need = int(lib.pkv_decode_workspace_bytes(B, Hq, D, 0))
    if workspace is None:
        with torch.cuda.device(dev):
            workspace = _workspace(dev, need)
    _check_cuda("workspace", workspace, device=dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = lib.pkv_paged_decode_attention_append(_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                                 _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                                 _ptr(seq_lens), B, Hq, Hkv, D, BS, NB, float(scale),
                                                 _dtype_code(q), _ptr(workspace),
                                                 workspace.numel() * workspace.element_size(), _ptr(status),
                                                 _stream(dev))
    _raise("pkv_paged_decode_attention_append", code)
    return out


def sample_workspace_bytes(B: int, V: int) -> int:
    return int(load_library().pkv_sample_workspace_bytes(B, V))


def sample_tokens(logits, temperature, top_k, top_p, seeds, offsets, tokens=None, status=None, min_p=None):
    """One token per row of logits [B, V] (float32); returns tokens [B] int32.

    seeds / offsets are int64 tensors holding uint64 bit patterns; min_p
    (float32 [B], optional) adds the min-p filter after top-p."""
    B, V = logits.shape
    dev = logits.device
    _check_cuda("logits", logits, torch.float32)
    _check_cuda("temperature", temperature, torch.float32, (B,), dev)
    _check_cuda("top_k", top_k, torch.int32, (B,), dev)
    _check_cuda("top_p", top_p, torch.float32, (B,), dev)
    if seeds.dtype not in (torch.int64, torch.uint64) or offsets.dtype not in (torch.int64, torch.uint64):
        raise TypeError("seeds and offsets must be 64-bit integer tensors")
    _check_cuda("seeds", seeds, shape=(B,), device=dev)
    _check_cuda("offsets", offsets, shape=(B,), device=dev)
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int32, device=dev)
    _check_cuda("tokens", tokens, torch.int32, (B,), dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    if min_p is not None:
        _check_cuda("min_p", min_p, torch.float32, (B,), dev)
        code = load_library().pkv_sample_tokens_ex(_ptr(tokens), _ptr(logits), B, V, _ptr(temperature),
                                                   _ptr(top_k), _ptr(top_p), _ptr(min_p), _ptr(seeds),
                                                   _ptr(offsets), _ptr(status), _stream(dev))
        _raise("pkv_sample_tokens_ex", code)
        return tokens
    code = load_library().pkv_sample_tokens(_ptr(tokens), _ptr(logits), B, V, _ptr(temperature),
                                            _ptr(top_k), _ptr(top_p), _ptr(seeds), _ptr(offsets),
                                            None, 0, _ptr(status), _stream(dev))
    _raise("pkv_sample_tokens", code)
    return tokens


class DecodeStep:
    """One decode step bound to fixed device buffers: the new token's K/V
    appended through the block table, paged decode attention
    (pkv_paged_decode_attention_append) and the sampler (pkv_sample_tokens, or
    pkv_sample_tokens_ex with min_p).  The buffers are checked once, here;
    run() passes the prepared pointers straight to the two C calls, so a
    serving loop pays a few microseconds of host time per step instead of
    re-validating every tensor.  The tensors must stay alive, in place and of
    the same shapes while the object is used (refill them in place between
    steps).  Returns the tokens tensor from run()."""

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, logits, temperature, top_k,
                 top_p, seeds, offsets, out=None, tokens=None, workspace=None, status=None, min_p=None,
                 scale: float = 0.0, stream=None):
        B, Hq, D = q.shape
        NB, Hkv, BS, D2 = k_cache.shape
        dev = q.device
        if D2 != D:
            raise ValueError("head_dim of q and the cache differ")
        _check_cuda("q", q)
        _check_cuda("k_cache", k_cache, q.dtype, device=dev)
        _check_cuda("v_cache", v_cache, q.dtype, k_cache.shape, dev)
        _check_cuda("k_new", k_new, q.dtype, (B, Hkv, D), dev)
        _check_cuda("v_new", v_new, q.dtype, (B, Hkv, D), dev)
        _check_cuda("block_tables", block_tables, torch.int32, device=dev)
        _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
        if block_tables.dim() != 2 or block_tables.shape[0] != B:
            raise ValueError("block_tables must be [B, max_blocks_per_seq]")
        if logits.dim() != 2 or logits.shape[0] != B:
            raise ValueError("logits must be [B, V]")
        V = logits.shape[1]
        _check_cuda("logits", logits, torch.float32, device=dev)
        _check_cuda("temperature", temperature, torch.float32, (B,), dev)
        _check_cuda("top_k", top_k, torch.int32, (B,), dev)
        _check_cuda("top_p", top_p, torch.float32, (B,), dev)
        if seeds.dtype not in (torch.int64, torch.uint64) or offsets.dtype not in (torch.int64, torch.uint64):
            raise TypeError("seeds and offsets must be 64-bit integer tensors")
        _check_cuda("seeds", seeds, shape=(B,), device=dev)
        _check_cuda("offsets", offsets, shape=(B,), device=dev)
        if min_p is not None:
            _check_cuda("min_p", min_p, torch.float32, (B,), dev)
        self.out = torch.empty_like(q) if out is None else out
        _check_cuda("out", self.out, q.dtype, q.shape, dev)
        self.tokens = torch.empty(B, dtype=torch.int32, device=dev) if tokens is None else tokens
        _check_cuda("tokens", self.tokens, torch.int32, (B,), dev)
        lib = load_library()
        need = int(lib.pkv_decode_workspace_bytes(B, Hq, D, 0))
        self.workspace = (torch.empty(max(need, 16), dtype=torch.uint8, device=dev) if workspace is None
                          else workspace)
        _check_cuda("workspace", self.workspace, device=dev)
        ws_bytes = self.workspace.numel() * self.workspace.element_size()
        if ws_bytes < need:
            raise ValueError(f"workspace holds {ws_bytes} bytes, the call needs {need}")
        if status is not None:
            _check_cuda("status", status, torch.int32, (1,), dev)
        self.status = status
        # keep every bound tensor referenced for the object's lifetime
        self._keep = (q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, logits, temperature, top_k,
                      top_p, seeds, offsets, min_p)
        self._dev = dev
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        sp = ctypes.c_void_p(s.cuda_stream)
        self._attn_fn = lib.pkv_paged_decode_attention_append
        self._attn = [_ptr(self.out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                      _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), B, Hq, Hkv, D, BS, NB,
                      ctypes.c_float(float(scale)), _dtype_code(q), _ptr(self.workspace), ws_bytes,
                      _ptr(status), sp]
        if min_p is None:
            self._samp_fn, self._samp_name = lib.pkv_sample_tokens, "pkv_sample_tokens"
            self._samp = [_ptr(self.tokens), _ptr(logits), B, V, _ptr(temperature), _ptr(top_k), _ptr(top_p),
                          _ptr(seeds), _ptr(offsets), None, 0, _ptr(status), sp]
        else:
            self._samp_fn, self._samp_name = lib.pkv_sample_tokens_ex, "pkv_sample_tokens_ex"
            self._samp = [_ptr(self.tokens), _ptr(logits), B, V, _ptr(temperature), _ptr(top_k), _ptr(top_p),
                          _ptr(min_p), _ptr(seeds), _ptr(offsets), _ptr(status), sp]

    def set_stream(self, stream) -> None:
        """Enqueue later steps on `stream` (a torch.cuda.Stream)."""
        sp = ctypes.c_void_p(stream.cuda_stream)
        self._attn[-1] = sp
        self._samp[-1] = sp

    def run_attention(self) -> torch.Tensor:
        """The append and the attention only; returns out."""
        code = self._attn_fn(*self._attn)
        if code != 0:
            raise PkvError("pkv_paged_decode_attention_append", code)
        return self.out

    def run_sampler(self) -> torch.Tensor:
        """The sampler only; returns the tokens."""
        code = self._samp_fn(*self._samp)
        if code != 0:
            raise PkvError(self._samp_name, code)
        return self.tokens

    def run(self) -> torch.Tensor:
        """The whole step; returns the tokens."""
        self.run_attention()
        return self.run_sampler()


def sample_tokens_typical(logits, temperature, typical_p, seeds, offsets, tokens=None, status=None):
    """Typical sampling: one token per row of logits [B, V] (float32); returns
    tokens [B] int32.  typical_p is float32 [B]; seeds / offsets as in
    sample_tokens."""
    B, V = logits.shape
    dev = logits.device
    _check_cuda("logits", logits, torch.float32)
    _check_cuda("temperature", temperature, torch.float32, (B,), dev)
    _check_cuda("typical_p", typical_p, torch.float32, (B,), dev)
    if seeds.dtype not in (torch.int64, torch.uint64) or offsets.dtype not in (torch.int64, torch.uint64):
        raise TypeError("seeds and offsets must be 64-bit integer tensors")
    _check_cuda("seeds", seeds, shape=(B,), device=dev)
    _check_cuda("offsets", offsets, shape=(B,), device=dev)
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int32, device=dev)
    _check_cuda("tokens", tokens, torch.int32, (B,), dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_sample_tokens_typical(_ptr(tokens), _ptr(logits), B, V, _ptr(temperature),
                                                    _ptr(typical_p), _ptr(seeds), _ptr(offsets), _ptr(status),
                                                    _stream(dev))
    _raise("pkv_sample_tokens_typical", code)
    return tokens


def copy_blocks(k_cache, v_cache, src, dst, status=None):
    """Copy physical block src[i] onto dst[i] in both pools (copy-on-write);
    src / dst are int32 device tensors of equal length."""
    NB, Hkv, BS, D = k_cache.shape
    dev = k_cache.device
    _check_cuda("k_cache", k_cache)
    _check_cuda("v_cache", v_cache, k_cache.dtype, k_cache.shape, dev)
    n = src.shape[0]
    _check_cuda("src", src, torch.int32, (n,), dev)
    _check_cuda("dst", dst, torch.int32, (n,), dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst), n, Hkv, D, BS, NB,
                                          _dtype_code(k_cache), _ptr(status), _stream(dev))
    _raise("pkv_copy_blocks", code)


class BlockPool:
    """Host-side reference-counted allocator of physical KV block ids (the
    library's pkv_block_pool).  Sequences are named by int ids."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        self._lib = load_library()
        self._p = self._lib.pkv_block_pool_create(num_blocks, block_size, max_blocks_per_seq)
        if not self._p:
            raise PkvError("pkv_block_pool_create", 1)
        self.num_blocks, self.block_size, self.max_blocks_per_seq = num_blocks, block_size, max_blocks_per_seq

    def close(self):
        if self._p:
            self._lib.pkv_block_pool_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, seq: int, length: int):
        _raise("pkv_seq_add", self._lib.pkv_seq_add(self._p, seq, length))

    def fork(self, parent: int, child: int):
        _raise("pkv_seq_fork", self._lib.pkv_seq_fork(self._p, parent, child))

    def append(self, seq: int):
        """Reserve the next token's slot; returns the copy-on-write pair
        (src, dst) or None."""
        s, d, n = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int()
        _raise("pkv_seq_append", self._lib.pkv_seq_append(self._p, seq, ctypes.byref(s), ctypes.byref(d),
                                                             ctypes.byref(n)))
        return (s.value, d.value) if n.value else None

    def free(self, seq: int):
        _raise("pkv_seq_free", self._lib.pkv_seq_free(self._p, seq))

    def length(self, seq: int) -> int:
        return int(self._lib.pkv_seq_length(self._p, seq))

    def num_free(self) -> int:
        return int(self._lib.pkv_block_pool_num_free(self._p))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_block_pool_refcount(self._p, block))

    def tables(self, seqs):
        """(block_tables int32 [n, max_blocks_per_seq], seq_lens int32 [n]) as CPU tensors."""
        n = len(seqs)
        ids = (ctypes.c_int64 * max(1, n))(*seqs)
        bt = torch.empty((n, self.max_blocks_per_seq), dtype=torch.int32)
        sl = torch.empty((n,), dtype=torch.int32)
        _raise("pkv_block_tables", self._lib.pkv_block_tables(self._p, ids, n, ctypes.c_void_p(bt.data_ptr()),
                                                               ctypes.c_void_p(sl.data_ptr())))
        return bt, sl


def spec_verify_workspace_bytes(B: int, gamma: int) -> int:
    return int(load_library().pkv_spec_verify_workspace_bytes(B, gamma))


def spec_verify(target_logits, draft_logits, draft_tokens, seq_lens, temperature, seeds, offsets,
                workspace=None, status=None):
    """Speculative verification of B requests with gamma drafts each.

    target_logits [B, gamma+1, V] float32, draft_logits [B, gamma, V] float32,
    draft_tokens [B, gamma] int32, seq_lens [B] int32 (including the drafts'
    KV), temperature [B] float32, seeds / offsets [B] 64-bit.  Returns
    (tokens [B, gamma+1] int32, n_accepted [B] int32, seq_lens_out [B] int32)."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    dev = target_logits.device
    _check_cuda("target_logits", target_logits, torch.float32)
    _check_cuda("draft_logits", draft_logits, torch.float32, (B, gamma, V), dev)
    _check_cuda("draft_tokens", draft_tokens, torch.int32, (B, gamma), dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    _check_cuda("temperature", temperature, torch.float32, (B,), dev)
    if seeds.dtype not in (torch.int64, torch.uint64) or offsets.dtype not in (torch.int64, torch.uint64):
        raise TypeError("seeds and offsets must be 64-bit integer tensors")
    _check_cuda("seeds", seeds, shape=(B,), device=dev)
    _check_cuda("offsets", offsets, shape=(B,), device=dev)
    lib = load_library()
    need = int(lib.pkv_spec_verify_workspace_bytes(B, gamma))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, device=dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
    n_acc = torch.empty((B,), dtype=torch.int32, device=dev)
    sl_out = torch.empty((B,), dtype=torch.int32, device=dev)
    code = lib.pkv_spec_verify(_ptr(tokens), _ptr(n_acc), _ptr(sl_out), _ptr(target_logits), _ptr(draft_logits),
                               _ptr(draft_tokens), _ptr(seq_lens), B, gamma, V, _ptr(temperature), _ptr(seeds),
                               _ptr(offsets), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _ptr(status), _stream(dev))
    _raise("pkv_spec_verify", code)
    return tokens, n_acc, sl_out


def apply_logits_processors(logits, allow_mask=None, row_ptr=None, tokens=None, counts=None, repetition=None,
                            frequency=None, presence=None, status=None):
    """Constraint mask (uint32 [B, ceil(V/32)], set bit = allowed) and CSR
    repetition / frequency / presence penalties, in place on logits [B, V]."""
    B, V = logits.shape
    dev = logits.device
    _check_cuda("logits", logits, torch.float32)
    if allow_mask is not None:
        if allow_mask.dtype not in (torch.int32, torch.uint32):
            raise TypeError("allow_mask must hold 32-bit words")
        _check_cuda("allow_mask", allow_mask, shape=(B, (V + 31) // 32), device=dev)
    if row_ptr is not None:
        _check_cuda("row_ptr", row_ptr, torch.int32, (B + 1,), dev)
        _check_cuda("tokens", tokens, torch.int32, device=dev)
        _check_cuda("counts", counts, torch.int32, tokens.shape, dev)
    for name, t in (("repetition", repetition), ("frequency", frequency), ("presence", presence)):
        if t is not None:
            _check_cuda(name, t, torch.float32, (B,), dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_apply_logits_processors(_ptr(logits), B, V, _ptr(allow_mask), _ptr(row_ptr),
                                                      _ptr(tokens), _ptr(counts), _ptr(repetition),
                                                      _ptr(frequency), _ptr(presence), _ptr(status), _stream(dev))
    _raise("pkv_apply_logits_processors", code)
    return logits


def kv_append_chunk(k_new, v_new, k_cache, v_cache, block_tables, seq_lens, q_start, status=None):
    """Append n_b = q_start[b+1] - q_start[b] rows of k_new / v_new [T_new, Hkv, D]
    per sequence at positions seq_lens[b] - n_b .. seq_lens[b] - 1."""
    NB, Hkv, BS, D = k_cache.shape
    B = seq_lens.shape[0]
    T = k_new.shape[0]
    dev = k_cache.device
    _check_cuda("k_cache", k_cache)
    _check_cuda("v_cache", v_cache, k_cache.dtype, k_cache.shape, dev)
    _check_cuda("k_new", k_new, k_cache.dtype, (T, Hkv, D), dev)
    _check_cuda("v_new", v_new, k_cache.dtype, (T, Hkv, D), dev)
    _check_cuda("block_tables", block_tables, torch.int32, device=dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    _check_cuda("q_start", q_start, torch.int32, (B + 1,), dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_kv_append_chunk(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                              _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                              _ptr(q_start), B, T, Hkv, D, BS, NB, _dtype_code(k_cache),
                                              _ptr(status), _stream(dev))
    _raise("pkv_kv_append_chunk", code)


def paged_prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, q_start, out=None, scale: float = 0.0,
                            status=None):
    """Causal attention of the packed chunk queries q [T_new, Hq, D]; returns out [T_new, Hq, D]."""
    T, Hq, D = q.shape
    NB, Hkv, BS, D2 = k_cache.shape
    B = seq_lens.shape[0]
    dev = q.device
    if D2 != D:
        raise ValueError("head_dim of q and the cache differ")
    _check_cuda("q", q)
    _check_cuda("k_cache", k_cache, q.dtype, device=dev)
    _check_cuda("v_cache", v_cache, q.dtype, k_cache.shape, dev)
    _check_cuda("block_tables", block_tables, torch.int32, device=dev)
    _check_cuda("seq_lens", seq_lens, torch.int32, (B,), dev)
    _check_cuda("q_start", q_start, torch.int32, (B + 1,), dev)
    if out is None:
        out = torch.empty_like(q)
    _check_cuda("out", out, q.dtype, q.shape, dev)
    if status is not None:
        _check_cuda("status", status, torch.int32, (1,), dev)
    code = load_library().pkv_paged_prefill_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                      _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                                      _ptr(q_start), B, T, Hq, Hkv, D, BS, NB, float(scale),
                                                      _dtype_code(q), _ptr(status), _stream(dev))
    _raise("pkv_paged_prefill_attention", code)
    return out
