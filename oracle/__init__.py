"""Float64 CPU oracle for scaled dot-product attention.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The CUDA library never
imports this package and this package never imports the CUDA library.

The arithmetic lives in ``attention_oracle.c`` (plain C, float64, one query
row at a time, three stages: scores, max-subtracted softmax, weighted sum of
V).  This module only compiles that file with gcc and marshals numpy arrays.

Citations for each stage are in the C file's header: "第 11 章 · Attention
入门" §11.1/§11.3/§11.8.1 and "3.3 Self-Attention机制深入理解" §3, §7.2, §9.3,
§10.2.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so``; return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleLib:
    """A loaded copy of the C oracle (``path`` defaults to the built library)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        fn = lib.attn_oracle_f64_window
        fn.restype = ctypes.c_int
        fn.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_int,
        ]
        self._lib = lib
        self.path = path

    def attention_f64(self, q, k, v, causal: bool, scale: float | None = None,
                      rows=None, nthreads: int | None = None, window: int = 0):
        """Return ``(o, lse)`` in float64.

        q: [B, Hq, Tq, D]; k, v: [B, Hkv, Tk, D] (numpy or CPU torch, any
        float dtype; values are widened to float32, which is exact for
        bf16/fp16/fp32).  ``scale`` defaults to 1/sqrt(D) ("第 11 章 ·
        Attention 入门" §11.1).  ``rows``: optional flat row indices
        ``(b*Hq + h)*Tq + i``; then ``o`` is [len(rows), D] and ``lse`` is
        [len(rows)].  Otherwise ``o`` is [B, Hq, Tq, D] and ``lse`` is
        [B, Hq, Tq].  ``lse`` is the natural-log log-sum-exp of the scaled,
        masked scores.  ``window`` > 0 (causal only) keeps, for each row, only
        the most recent ``window`` keys up to its causal limit ("第 11 章 ·
        Attention 入门" §11.8.4, Sliding Window Attention).
        """
        q = _as_f32(q)
        k = _as_f32(k)
        v = _as_f32(v)
        if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
            raise ValueError("q, k, v must be 4-D [B, H, T, D]")
        B, Hq, Tq, D = q.shape
        Bk, Hkv, Tk, Dk = k.shape
        if k.shape != v.shape or Bk != B or Dk != D:
            raise ValueError("shape mismatch between q, k and v")
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        if rows is not None:
            rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
            n = rows.shape[0]
            o = np.empty((n, D), dtype=np.float64)
            lse = np.empty((n,), dtype=np.float64)
            rows_ptr, nrows = rows.ctypes.data, n
        else:
            o = np.empty((B, Hq, Tq, D), dtype=np.float64)
            lse = np.empty((B, Hq, Tq), dtype=np.float64)
            rows_ptr, nrows = None, 0
        rc = self._lib.attn_oracle_f64_window(
            q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, Hkv, Tq, Tk, D,
            1 if causal else 0, int(window), float(scale), rows_ptr, nrows, o.ctypes.data,
            lse.ctypes.data, int(nthreads or default_threads()))
        if rc != 0:
            raise ValueError(f"attn_oracle_f64 failed with code {rc}")
        return o, lse


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = OracleLib(_LIB_PATH)
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def attention_f64(q, k, v, causal: bool, scale: float | None = None,
                  rows=None, nthreads: int | None = None, window: int = 0):
    """Float64 attention of the built oracle; see ``OracleLib.attention_f64``."""
    return _load().attention_f64(q, k, v, causal, scale, rows, nthreads, window)


def decode_paged_f64(q, kv_cache, block_table, seq_lens, scale: float | None = None,
                     nthreads: int | None = None):
    """Float64 decode attention over a paged KV cache; returns ``(o, lse)``.

    The cache is a pool of physical blocks of ``page_size`` tokens, each
    holding the K and the V rows of those tokens for every KV head
    ("第 11 章 · Attention 入门", 11.11, the KV-cache / VMM passage: a block
    holds N tokens' K + V for all KV heads, and ``block_table[req][t/16]``
    names the physical block of token t of request req).

    q: [B, Hq, D] or [B, Hq, 1, D]; kv_cache: [num_blocks, 2, Hkv, page_size,
    D] (index 0 = K, 1 = V); block_table: [B, max_pages] integers;
    seq_lens: [B] keys of each request.  The decode query sees all of its
    request's keys.  Request b's keys are gathered token by token, t ->
    block ``block_table[b, t // page_size]``, row ``t % page_size``, and the
    plain attention of the dense oracle is taken over them.  A request with
    no keys gets O = 0 and lse = -inf (its softmax is over an empty set).
    o: [B, Hq, D]; lse: [B, Hq].
    """
    q = _as_f32(q)
    if q.ndim == 4:
        if q.shape[2] != 1:
            raise ValueError("paged decode takes one query row per head")
        q = q[:, :, 0, :]
    kv = _as_f32(kv_cache)
    bt = np.asarray(block_table.cpu() if hasattr(block_table, "cpu") else block_table,
                    dtype=np.int64)
    sl = np.asarray(seq_lens.cpu() if hasattr(seq_lens, "cpu") else seq_lens, dtype=np.int64)
    if kv.ndim != 5 or kv.shape[1] != 2:
        raise ValueError("kv_cache must be [num_blocks, 2, Hkv, page_size, D]")
    B, Hq, D = q.shape
    nblk, _, Hkv, P, Dk = kv.shape
    if Dk != D or bt.shape[0] != B or sl.shape[0] != B:
        raise ValueError("shape mismatch")
    o = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(sl[b])
        if L < 0 or L > bt.shape[1] * P:
            raise ValueError("sequence length outside the block table")
        if L == 0:
            continue
        t = np.arange(L)
        blk = bt[b, t // P]
        if (blk < 0).any() or (blk >= nblk).any():
            raise ValueError("block id out of range")
        k = kv[blk, 0, :, t % P, :]  # [L, Hkv, D]
        v = kv[blk, 1, :, t % P, :]
        k = np.ascontiguousarray(k.transpose(1, 0, 2))[None]  # [1, Hkv, L, D]
        v = np.ascontiguousarray(v.transpose(1, 0, 2))[None]
        ob, lb = attention_f64(q[b][None, :, None, :], k, v, False, scale, None, nthreads)
        o[b] = ob[0, :, 0, :]
        lse[b] = lb[0, :, 0]
    return o, lse


def attention_varlen_f64(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool,
                         scale: float | None = None, window: int = 0,
                         seqs=None, nthreads: int | None = None):
    """Float64 attention over sequences packed along the token axis; returns
    ``(o, lse)``.

    q: [total_q, Hq, D]; k, v: [total_k, Hkv, D] (the (T, H, D) layout of
    "第 11 章 · Attention 入门", 11.11).  Sequence b owns query rows
    ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1`` and key rows
    ``cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1``; it is the plain attention of
    the dense oracle over those rows alone, with the causal mask (and
    ``window``) aligned to the end of its keys as in the dense oracle.  A
    sequence with query rows but no keys gets O = 0 and lse = -inf (its
    softmax is over an empty set).  ``seqs``: optional sequence indices to
    compute; the others stay O = 0, lse = NaN.
    o: [total_q, Hq, D]; lse: [Hq, total_q].
    """
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    cq = np.asarray(cu_seqlens_q.cpu() if hasattr(cu_seqlens_q, "cpu") else cu_seqlens_q,
                    dtype=np.int64)
    ck = np.asarray(cu_seqlens_k.cpu() if hasattr(cu_seqlens_k, "cpu") else cu_seqlens_k,
                    dtype=np.int64)
    if q.ndim != 3 or k.ndim != 3 or k.shape != v.shape or q.shape[2] != k.shape[2]:
        raise ValueError("q must be [total_q, Hq, D] and k, v [total_k, Hkv, D]")
    if cq.ndim != 1 or cq.shape != ck.shape or cq.shape[0] < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must be [B + 1]")
    TQ, Hq, D = q.shape
    TK, Hkv, _ = k.shape
    B = cq.shape[0] - 1
    if (np.diff(cq) < 0).any() or cq[0] < 0 or cq[-1] > TQ:
        raise ValueError("cu_seqlens_q is not a non-decreasing offset list inside q")
    if (np.diff(ck) < 0).any() or ck[0] < 0 or ck[-1] > TK:
        raise ValueError("cu_seqlens_k is not a non-decreasing offset list inside k")
    o = np.zeros((TQ, Hq, D), dtype=np.float64)
    lse = np.full((Hq, TQ), np.nan, dtype=np.float64)
    for b in (range(B) if seqs is None else seqs):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        if k1 == k0:
            lse[:, q0:q1] = -np.inf
            continue
        if causal and q1 - q0 > k1 - k0:
            raise ValueError("causal sequence with more queries than keys")
        qb = np.ascontiguousarray(q[q0:q1].transpose(1, 0, 2))[None]  # [1, Hq, Tq, D]
        kb = np.ascontiguousarray(k[k0:k1].transpose(1, 0, 2))[None]  # [1, Hkv, Tk, D]
        vb = np.ascontiguousarray(v[k0:k1].transpose(1, 0, 2))[None]
        ob, lb = attention_f64(qb, kb, vb, causal, scale, None, nthreads, window)
        o[q0:q1] = ob[0].transpose(1, 0, 2)
        lse[:, q0:q1] = lb[0]
    return o, lse


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch  # local: torch is optional for numpy callers
        x = x.to(torch.float32).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))
