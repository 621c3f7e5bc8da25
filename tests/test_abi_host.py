"""Host-side checks of the C ABI (no GPU needed, no kernel is launched):
the library builds, loads and exports every declared entry point, and
argument validation rejects bad calls before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from transformer_attention_fwd_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    names = []
    for h in ("attn.h", "attn_diag.h"):
        text = open(os.path.join(ROOT, "include", h), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:attn_status|const char\*|void)\s+(attn_\w+)\s*\(", text, re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_prefill", "attn_fwd_decode", "attn_fwd_decode_paged",
            "attn_fwd_window", "attn_fwd_varlen", "attn_fwd_host",
            "attn_get_device_status", "attn_last_error", "attn_diag_mma_tile",
            "attn_diag_wait_timeout"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def _fwd(lib):
    f = lib.attn_fwd
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    lib.attn_last_error.restype = ctypes.c_char_p
    return f


FAKE = 0x10000  # aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("args,code,msg", [
    ((0, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 64, 1, 0.125, 1), 1, "non-null"),
    ((FAKE + 2, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 64, 1, 0.125, 1), 1, "aligned"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE + 1, 1, 1, 1, 4, 4, 64, 1, 0.125, 1), 1, "lse"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 3, 2, 4, 4, 64, 1, 0.125, 1), 1, "multiple"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 96, 1, 0.125, 1), 2, "D=96"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 8, 4, 64, 1, 0.125, 1), 1, "Tq <= Tk"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 64, 0, 0.0, 1), 1, "scale"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 64, 0, float("nan"), 1), 1, "scale"),
    ((FAKE, FAKE, FAKE, FAKE, None, 0, 1, 1, 4, 4, 64, 0, 0.125, 1), 1, ">= 1"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 0, 4, 64, 0, 0.125, 1), 1, ">= 1"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 64, 0, 0.125, 7), 1, "dtype"),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 4, 4, 96, 1, 0.125, 2), 2, "D=96"),   # fp16
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 1, 1, 8, 4, 64, 1, 0.125, 2), 1, "Tq <= Tk"),  # fp16
])
def test_invalid_arguments_rejected_before_launch(lib, args, code, msg):
    f = _fwd(lib)
    assert f(*args, None) == code
    assert msg in lib.attn_last_error().decode()


def test_decode_split_count_range(lib):
    f = lib.attn_fwd_decode
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 128, 128, 0.1, 300, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 128, 128, 0.1, -1, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 3, 128, 128, 0.1, 0, None) == 1


@pytest.mark.parametrize("args,code,msg", [
    # q, kv, block_table, seq_lens, o, lse, B, Hq, Hkv, D, page, max_pages, num_blocks, scale
    ((0, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 8, 0.1), 1, "non-null"),
    ((FAKE, FAKE, 0, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 8, 0.1), 1, "non-null"),
    ((FAKE, FAKE + 8, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 8, 0.1), 1, "16-byte"),
    ((FAKE, FAKE, FAKE + 2, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 8, 0.1), 1, "4-byte"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 3, 128, 16, 4, 8, 0.1), 1, "multiple"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 80, 16, 4, 8, 0.1), 2, "D=80"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 0, 4, 8, 0.1), 1, ">= 1"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 0, 8, 0.1), 1, ">= 1"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 0, 0.1), 1, ">= 1"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 16, 4, 8, -1.0), 1, "scale"),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 128, 1 << 20, 1 << 12, 8, 0.1), 1, "2^31"),
])
def test_paged_decode_arguments_rejected_before_launch(lib, args, code, msg):
    f = lib.attn_fwd_decode_paged
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    lib.attn_last_error.restype = ctypes.c_char_p
    assert f(*args, 1, None) == code  # bf16
    assert f(*args, 2, None) == code  # fp16: the same checks
    assert msg in lib.attn_last_error().decode()


def test_host_call_arguments_rejected_before_launch(lib):
    f = lib.attn_fwd_host
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    lib.attn_last_error.restype = ctypes.c_char_p
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 1, 0.1, 9, None) == 1  # dtype
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 96, 1, 0.1, 1, None) == 2   # D
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 3, 64, 64, 128, 1, 0.1, 1, None) == 1  # GQA
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 80, 64, 128, 1, 0.1, 2, None) == 1  # Tq > Tk
    assert f(None, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 1, 0.1, 1, None) == 1


def test_window_arguments_rejected_before_launch(lib):
    f = lib.attn_fwd_window
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    lib.attn_last_error.restype = ctypes.c_char_p
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 0, 0.1, 1, None) == 1
    assert b"window" in lib.attn_last_error()
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 16, 0.1, 0, None) == 2  # fp32
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 80, 64, 128, 16, 0.1, 1, None) == 1  # Tq > Tk
    assert f(FAKE + 4, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 16, 0.1, 1, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 16, 0.1, 3, None) == 1  # dtype
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 64, 64, 128, 0, 0.1, 2, None) == 1  # fp16, W=0


def test_varlen_arguments_rejected_before_launch(lib):
    f = lib.attn_fwd_varlen
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P]
    f.restype = ctypes.c_int
    lib.attn_last_error.restype = ctypes.c_char_p

    def call(q=FAKE, cu=FAKE, B=2, Hq=4, Hkv=2, tq=300, tk=300, D=128, causal=1, window=0,
             scale=0.1, dtype=1):
        return f(q, FAKE, FAKE, FAKE, None, cu, FAKE, B, Hq, Hkv, tq, tk, D, causal, window,
                 scale, dtype, None)

    assert call(causal=0, window=16) == 1 and b"causal" in lib.attn_last_error()
    assert call(window=-1) == 1
    assert call(D=96) == 2
    assert call(Hq=6, Hkv=4) == 1
    assert call(tq=-1) == 1
    assert call(scale=0.0) == 1
    assert call(q=FAKE + 4) == 1
    assert call(cu=None) == 1
    assert call(dtype=0) == 2  # fp32 is not packed
    assert call(dtype=5) == 1
    assert call(D=96, dtype=2) == 2
    assert call(B=0) == 1
    # No query rows: nothing to launch, no device needed.
    assert call(q=None, tq=0) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    from transformer_attention_fwd_gb300 import attn as a  # noqa: F401  (loads the built lib)
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "attn_copy", os.path.join(ROOT, "transformer_attention_fwd_gb300", "attn.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with pytest.raises(RuntimeError, match="missing"):
        mod._load(str(tmp_path / "libattn.so"))
