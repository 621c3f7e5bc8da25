"""Shared helpers for the GPU parity tests (marked ``gpu``)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

# Tolerances (max abs error against the float64 oracle on the same inputs).
TOL_O_F32 = 1e-5      # fp32 I/O
TOL_LSE_F32 = 1e-5
TOL_O_BF16 = 1e-2     # bf16 I/O, fp32 accumulation
TOL_LSE_BF16 = 1e-4


def attn():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for tests marked gpu")
    from transformer_attention_fwd_gb300 import build
    build.build()
    from transformer_attention_fwd_gb300 import attn as a
    return a


def to_dev(*ts):
    return [t.cuda().contiguous() for t in ts]


def check_status(a):
    st = a.device_status()
    assert st == a.ATTN_OK, f"device status {st}: {a.last_error()}"


def compare(o_gpu, lse_gpu, o_ref, lse_ref, tol_o, tol_lse, what=""):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    err_o = float(np.abs(o - o_ref).max()) if o.size else 0.0
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    assert err_o <= tol_o, f"{what}: max |O - O_ref| = {err_o:.3e} > {tol_o:.1e}"
    if lse_gpu is not None and lse_ref is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        err_l = float(np.abs(l - lse_ref).max()) if l.size else 0.0
        assert err_l <= tol_lse, f"{what}: max |lse - lse_ref| = {err_l:.3e} > {tol_lse:.1e}"
        return err_o, err_l
    return err_o, None


def sample_rows(B, Hq, Tq, n, seed=0):
    """Flat row indices covering the first/last rows of every head, tile
    boundaries (multiples of 128 +-1) and random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for bh in range(B * Hq):
        for i in (0, 1, Tq - 1, Tq // 2):
            rows.add(bh * Tq + i)
    for t in range(128, Tq, 128):
        for i in (t - 1, t):
            bh = int(rng.integers(0, B * Hq))
            rows.add(bh * Tq + i)
    while len(rows) < n:
        rows.add(int(rng.integers(0, B * Hq * Tq)))
    return np.array(sorted(rows), dtype=np.int64)
