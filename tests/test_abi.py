"""The C-ABI library builds for sm_103a, loads, and exports every declared entry point.

No compute call is made here (no GPU needed): only host-side behaviour --
symbol export, status strings, pure-host workspace sizing and argument checks
that return before anything is launched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_table_gb300 import build as B
    B.build()
    import paged_kv_decode_table_gb300 as pkv
    return pkv.load_library()


def _declared_symbols():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert {"pkv_kv_append", "pkv_paged_decode_attention", "pkv_sample_tokens"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    import paged_kv_decode_table_gb300 as pkv
    for code, name in pkv.STATUS.items():
        assert pkv.status_string(code) == name
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"
    assert lib.pkv_version() >= 100


def test_workspace_sizing_is_host_arithmetic(lib):
    import paged_kv_decode_table_gb300 as pkv
    a = pkv.decode_workspace_bytes(64, 32, 128, num_sms=152)
    b = pkv.decode_workspace_bytes(64, 32, 128, num_sms=76)
    assert a > b > 0
    # partial slots: (B + P) x Hq x (D + 2) floats plus the schedule
    assert a >= (64 + 152) * 32 * (128 + 2) * 4
    assert a % 256 == 0
    assert pkv.decode_workspace_bytes(0, 32, 128, num_sms=152) > 0
    assert pkv.decode_workspace_bytes(-1, 32, 128, num_sms=152) == 0
    assert pkv.sample_workspace_bytes(256, 152064) == 0


def test_argument_errors_return_before_launch(lib):
    P = ctypes.c_void_p
    # B == 0 is a no-op
    assert lib.pkv_kv_append(None, None, None, None, None, 1, None, 0, 1, 4, 4, 1, 0, None, None) == 0
    # null pointers, bad shapes, bad dtype
    assert lib.pkv_kv_append(None, None, None, None, None, 1, None, 2, 1, 4, 4, 1, 0, None, None) == 1
    assert lib.pkv_kv_append(P(16), P(16), P(16), P(16), P(16), 1, P(16), 2, 1, 4, 4, 1, 7, None, None) == 1
    assert lib.pkv_paged_decode_attention(None, None, None, None, None, 1, None, 2, 3, 2, 4, 4, 1, 0.0, 0,
                                          None, 0, None, None) == 1   # Hq % Hkv != 0
    assert lib.pkv_paged_decode_attention(None, None, None, None, None, 1, None, 2, 4, 2, 512, 4, 1, 0.0, 0,
                                          None, 0, None, None) == 1   # D too large
    assert lib.pkv_paged_decode_attention(None, None, None, None, None, 1, None, 0, 4, 2, 4, 4, 1, 0.0, 0,
                                          None, 0, None, None) == 0   # empty batch
    A = lib.pkv_paged_decode_attention_append
    assert A(None, None, None, None, None, None, None, 1, None, 2, 3, 2, 4, 4, 1, 0.0, 0,
             None, 0, None, None) == 1   # Hq % Hkv != 0
    assert A(None, None, None, None, None, None, None, 1, None, 0, 4, 2, 4, 4, 1, 0.0, 0,
             None, 0, None, None) == 0   # empty batch
    assert A(P(16), P(16), None, P(16), P(16), P(16), P(16), 1, P(16), 2, 4, 2, 4, 4, 1, 0.0, 0,
             P(16), 1 << 30, None, None) == 1   # k_new missing
    assert lib.pkv_sample_tokens(None, None, 4, 0, None, None, None, None, None, None, 0, None, None) == 1
    assert lib.pkv_sample_tokens(None, None, 4, 1 << 24, None, None, None, None, None, None, 0, None, None) == 1
    assert lib.pkv_sample_tokens(None, None, 0, 100, None, None, None, None, None, None, 0, None, None) == 0
    assert lib.pkv_sample_tokens_typical(None, None, 4, 100, None, None, None, None, None, None) == 1
    assert lib.pkv_sample_tokens_typical(None, None, 4, 1 << 24, None, None, None, None, None, None) == 1
    assert lib.pkv_sample_tokens_typical(None, None, 0, 100, None, None, None, None, None, None) == 0


def test_library_has_no_oracle_dependency():
    """The product library links nothing from oracle/ and the package never imports it."""
    pkg = os.path.join(ROOT, "paged_kv_decode_table_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pkv_oracle" not in text, f
