"""Causal attention with a sliding window ("第 11 章 · Attention 入门" §11.8.4,
Sliding Window Attention: only the most recent W tokens) against the float64
oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, sample_rows,
                      to_dev)
from transformer_attention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Tq,Tk,D,W", [
    (1000, 1000, 128, 1), (1000, 1000, 128, 64), (1000, 1000, 128, 127),
    (1000, 1000, 128, 128), (1000, 1000, 128, 129), (1000, 1000, 128, 300),
    (700, 700, 64, 200), (700, 700, 64, 256),
    (300, 1000, 128, 256),      # Tq < Tk: rows sit at positions 700..999
    (1, 777, 128, 100),         # one query row
    (515, 515, 64, 5000),       # window longer than the sequence
])
def test_window_matches_oracle(Tq, Tk, D, W):
    a = attn()
    q, k, v = make_qkv(2, 4, 2, Tq, Tk, D, "bf16", seed=71)
    o, lse = a.attn_fwd_window(*to_dev(q, k, v), W)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, True, window=W)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"Tq{Tq} Tk{Tk} D{D} W{W}")


def test_window_covering_all_keys_is_exactly_causal():
    a = attn()
    q, k, v = to_dev(*make_qkv(1, 8, 2, 600, 900, 128, "bf16", seed=72))
    o1, l1 = a.attn_fwd(q, k, v, causal=True)
    o2, l2 = a.attn_fwd_window(q, k, v, 900)
    check_status(a)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_window_of_one_returns_own_value_exactly():
    a = attn()
    q, k, v = make_qkv(1, 4, 4, 300, 300, 64, "bf16", seed=73)
    o, _ = a.attn_fwd_window(*to_dev(q, k, v), 1)
    check_status(a)
    assert torch.equal(o.cpu(), v)


def test_mistral_like_window_full_size_sampled():
    """Llama-3-8B shapes at T = 8192 with a 4096-token window (the page's
    Mistral figure): sampled rows, including tile and window edges."""
    a = attn()
    B, Hq, Hkv, T, D, W = 1, 32, 8, 8192, 128, 4096
    q, k, v = make_qkv(B, Hq, Hkv, T, T, D, "bf16", seed=74)
    o, lse = a.attn_fwd_window(*to_dev(q, k, v), W)
    check_status(a)
    rows = sample_rows(B, Hq, T, 1500, seed=5)
    extra = [h * T + i for h in range(0, Hq, 7) for i in (W - 2, W - 1, W, W + 1, W + 127, W + 128)]
    rows = np.unique(np.concatenate([rows, np.array(extra, dtype=np.int64)]))
    o_ref, lse_ref = oracle.attention_f64(q, k, v, True, rows=rows, window=W)
    og = o.reshape(-1, D)[torch.from_numpy(rows).cuda()]
    lg = lse.reshape(-1)[torch.from_numpy(rows).cuda()]
    compare(og, lg, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, "T8192 W4096")
