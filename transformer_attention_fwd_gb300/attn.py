"""ctypes binding over libattn.so (include/attn.h, include/attn_diag.h).

Argument marshalling only: the functions check tensor placement, dtype and
contiguity, allocate outputs with torch, and pass raw device pointers plus the
current CUDA stream to the C ABI.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  If the library is missing the
import-time load raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libattn.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_NO_MEMORY = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_BAD_INPUT = 6
ATTN_F32 = 0
ATTN_BF16 = 1
ATTN_F16 = 2

STATUS_NAMES = {
    ATTN_OK: "ATTN_OK", ATTN_ERR_INVALID_ARG: "ATTN_ERR_INVALID_ARG",
    ATTN_ERR_UNSUPPORTED: "ATTN_ERR_UNSUPPORTED", ATTN_ERR_CUDA: "ATTN_ERR_CUDA",
    ATTN_ERR_NO_MEMORY: "ATTN_ERR_NO_MEMORY", ATTN_ERR_TIMEOUT: "ATTN_ERR_TIMEOUT",
    ATTN_ERR_BAD_INPUT: "ATTN_ERR_BAD_INPUT",
}


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with transformer_attention_fwd_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I, F, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
    sig = {
        "attn_fwd": [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P],
        "attn_fwd_prefill": [P, P, P, P, P, I, I, I, I, I, I, I, F, P],
        "attn_fwd_decode": [P, P, P, P, P, I, I, I, I, I, F, I, P],
        "attn_fwd_decode_paged": [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P],
        "attn_fwd_window": [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P],
        "attn_fwd_host": [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P],
        "attn_fwd_varlen": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P],
        "attn_get_device_status": [P],
        "attn_diag_mma_tile": [P, P, P, P, P, I, P],
        "attn_diag_wait_timeout": [LL, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.attn_last_error.argtypes = []
    lib.attn_last_error.restype = ctypes.c_char_p
    lib.attn_last_launch_info.argtypes = [ctypes.POINTER(I)] * 3
    lib.attn_last_launch_info.restype = None
    return lib


lib = _load()


def last_error() -> str:
    return lib.attn_last_error().decode("utf-8", "replace")


def _check(status: int) -> None:
    if status != ATTN_OK:
        raise AttnError(status, last_error())


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def last_launch_info():
    g, i, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    lib.attn_last_launch_info(ctypes.byref(g), ctypes.byref(i), ctypes.byref(k))
    return g.value, i.value, k.value


def _check_buffer(name, t, shape, dtype, device):
    """A caller-supplied output buffer must hold exactly what the call writes:
    the kernels write through its pointer and know nothing of its size."""
    if t is None:
        return
    if t.device != torch.device(device):
        raise ValueError(f"{name} must be on {device} (got {t.device})")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != math.prod(shape):
        raise ValueError(f"{name} must hold {tuple(shape)} = {math.prod(shape)} elements "
                         f"(got {tuple(t.shape)})")


def _same_device(**tensors):
    """Every tensor on one CUDA device, the current one (the library launches
    on the current device)."""
    devs = {t.device for t in tensors.values()}
    if len(devs) != 1:
        raise ValueError(f"{', '.join(tensors)} must be on one device (got {sorted(map(str, devs))})")
    dev = devs.pop()
    if dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"tensors are on {dev} but the current device is "
                         f"cuda:{torch.cuda.current_device()}; call under torch.cuda.device({dev})")


def _shapes(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, H, T, D]")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [B, H, T, D]")
    _same_device(q=q, k=k, v=v)
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    B, Hq, Tq, D = q.shape
    Bk, Hkv, Tk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Hkv, Tk, D] with q's B and D")
    return B, Hq, Hkv, Tq, Tk, D


def _outputs(q, out, lse, want_lse):
    B, Hq, Tq, D = q.shape
    _check_buffer("out", out, q.shape, q.dtype, q.device)
    _check_buffer("lse", lse, (B, Hq, Tq), torch.float32, q.device)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    return o, lse


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             want_lse: bool = True, stream=None):
    """O = softmax(Q K^T * scale + causal mask) V through ``attn_fwd``.

    q: [B, Hq, Tq, D], k/v: [B, Hkv, Tk, D], all fp32, all bf16 or all fp16 CUDA
    tensors.
    Returns ``(o, lse)``; ``lse`` (fp32 [B, Hq, Tq]) is None if not wanted.
    ``scale`` defaults to 1/sqrt(D).
    """
    B, Hq, Hkv, Tq, Tk, D = _shapes(q, k, v)
    if q.dtype == torch.float32:
        dt = ATTN_F32
    elif q.dtype == torch.bfloat16:
        dt = ATTN_BF16
    elif q.dtype == torch.float16:
        dt = ATTN_F16
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o, lse = _outputs(q, out, lse, want_lse)
    _check(lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tk, D,
                        1 if causal else 0, scale, dt, _stream_handle(stream)))
    return o, lse


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                  lse=None, want_lse: bool = True, stream=None):
    """``attn_fwd`` on host tensors (``attn_fwd_host``): q [B, Hq, Tq, D] and
    k/v [B, Hkv, Tk, D] CPU tensors (fp32, bf16 or fp16; pinned memory lets
    the copies overlap the compute).  Returns CPU ``(o, lse)``, complete once
    ``stream`` (default: the current CUDA stream) has run the call."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
        if not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be contiguous [B, H, T, D]")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    dt = {torch.float32: ATTN_F32, torch.bfloat16: ATTN_BF16, torch.float16: ATTN_F16}.get(q.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, Hq, Tq, D = q.shape
    Bk, Hkv, Tk, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be [B, Hkv, Tk, D] with q's B and D")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check_buffer("out", out, q.shape, q.dtype, "cpu")
    _check_buffer("lse", lse, (B, Hq, Tq), torch.float32, "cpu")
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, pin_memory=pin)
    _check(lib.attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tk,
                             D, 1 if causal else 0, scale, dt, _stream_handle(stream)))
    return o, lse


def attn_fwd_prefill(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                     lse=None, want_lse: bool = True, stream=None):
    """The bf16 tensor-core path for any Tq (``attn_fwd_prefill``)."""
    B, Hq, Hkv, Tq, Tk, D = _shapes(q, k, v)
    if q.dtype != torch.bfloat16:
        raise ValueError("attn_fwd_prefill takes bf16 tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o, lse = _outputs(q, out, lse, want_lse)
    _check(lib.attn_fwd_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq,
                                Tk, D, 1 if causal else 0, scale, _stream_handle(stream)))
    return o, lse


def attn_fwd_decode(q, k, v, scale: float | None = None, num_splits: int = 0, out=None,
                    lse=None, want_lse: bool = True, stream=None):
    """Split-KV decode (``attn_fwd_decode``): q [B, Hq, 1, D] bf16 against
    k/v [B, Hkv, Tk, D]; ``num_splits`` 0 = automatic."""
    B, Hq, Hkv, Tq, Tk, D = _shapes(q, k, v)
    if Tq != 1:
        raise ValueError("decode takes one query row per (b, hq)")
    if q.dtype != torch.bfloat16:
        raise ValueError("attn_fwd_decode takes bf16 tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o, lse = _outputs(q, out, lse, want_lse)
    _check(lib.attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tk, D,
                               scale, int(num_splits), _stream_handle(stream)))
    return o, lse


def attn_fwd_window(q, k, v, window: int, scale: float | None = None, out=None, lse=None,
                    want_lse: bool = True, stream=None):
    """Causal attention with a sliding window of ``window`` keys
    (``attn_fwd_window``); bf16 [B, Hq, Tq, D] / [B, Hkv, Tk, D] CUDA tensors."""
    B, Hq, Hkv, Tq, Tk, D = _shapes(q, k, v)
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("attn_fwd_window takes bf16 or fp16 tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o, lse = _outputs(q, out, lse, want_lse)
    _check(lib.attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Tq, Tk,
                               D, int(window), scale,
                               ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16,
                               _stream_handle(stream)))
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool, window: int = 0,
                    scale: float | None = None, out=None, lse=None, want_lse: bool = True,
                    stream=None):
    """Attention over sequences packed along the token axis (``attn_fwd_varlen``).

    q: [total_q, Hq, D] bf16; k, v: [total_k, Hkv, D] bf16; cu_seqlens_q,
    cu_seqlens_k: [B + 1] int32 offsets; all CUDA tensors.  Returns
    ``(o [total_q, Hq, D], lse [Hq, total_q] or None)``.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("cu_seqlens_q", cu_seqlens_q),
                    ("cu_seqlens_k", cu_seqlens_k)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or q.shape[2] != k.shape[2]:
        raise ValueError("q must be [total_q, Hq, D] and k, v [total_k, Hkv, D]")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("attn_fwd_varlen takes bf16 or fp16 tensors")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be int32")
    if (cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape != cu_seqlens_k.shape
            or cu_seqlens_q.shape[0] < 2):
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be [B + 1]")
    _same_device(q=q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k)
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.shape[0] - 1
    _check_buffer("out", out, q.shape, q.dtype, q.device)
    _check_buffer("lse", lse, (Hq, total_q), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    _check(lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                               _ptr(cu_seqlens_k), B, Hq, Hkv, total_q, total_k, D,
                               1 if causal else 0, int(window), scale,
                               ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16,
                               _stream_handle(stream)))
    return o, lse


def attn_fwd_decode_paged(q, kv_cache, block_table, seq_lens, scale: float | None = None,
                          out=None, lse=None, want_lse: bool = True, stream=None):
    """Decode against a paged KV cache (``attn_fwd_decode_paged``).

    q: [B, Hq, 1, D] bf16; kv_cache: [num_blocks, 2, Hkv, page_size, D] bf16
    (0 = K, 1 = V); block_table: [B, max_pages] int32; seq_lens: [B] int32; all
    CUDA tensors.  Returns ``(o [B, Hq, 1, D], lse [B, Hq] or None)``.
    """
    for name, t in (("q", q), ("kv_cache", kv_cache), ("block_table", block_table),
                    ("seq_lens", seq_lens)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dim() != 4 or q.shape[2] != 1 or q.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("q must be bf16 or fp16 [B, Hq, 1, D]")
    if kv_cache.dim() != 5 or kv_cache.shape[1] != 2 or kv_cache.dtype != q.dtype:
        raise ValueError("kv_cache must be [num_blocks, 2, Hkv, page_size, D] in q's dtype")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    B, Hq, _, D = q.shape
    nblk, _, Hkv, page, Dk = kv_cache.shape
    if Dk != D or block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and seq_lens [B], with q's B and D")
    _same_device(q=q, kv_cache=kv_cache, block_table=block_table, seq_lens=seq_lens)
    _check_buffer("out", out, q.shape, q.dtype, q.device)
    _check_buffer("lse", lse, (B, Hq), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _check(lib.attn_fwd_decode_paged(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                                     _ptr(o), _ptr(lse), B, Hq, Hkv, D, page,
                                     block_table.shape[1], nblk, scale,
                                     ATTN_F16 if q.dtype == torch.float16 else ATTN_BF16,
                                     _stream_handle(stream)))
    return o, lse


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status as an
    attn_status code (ATTN_ERR_TIMEOUT if a kernel wait ran out of time,
    ATTN_ERR_BAD_INPUT if a kernel met an out-of-range device-side index)."""
    return lib.attn_get_device_status(_stream_handle(stream))


def diag_mma_tile(a, b, v, stream=None):
    """Self-test of the tensor-core tile products; returns (s, o) fp32."""
    D = a.shape[1]
    s = torch.empty((128, 128), dtype=torch.float32, device=a.device)
    o = torch.empty((128, D), dtype=torch.float32, device=a.device)
    _check(lib.attn_diag_mma_tile(_ptr(a), _ptr(b), _ptr(v), _ptr(s), _ptr(o), D,
                                  _stream_handle(stream)))
    return s, o


def diag_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib.attn_diag_wait_timeout(int(timeout_ns), _stream_handle(stream)))
