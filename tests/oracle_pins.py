"""Pins that tie the float64 oracle to what the pages and mathematics fix.

Every pin is a function ``pin_*(attention)`` that takes an oracle-shaped
callable ``attention(q, k, v, causal, scale=None, rows=None) -> (o, lse)``
and raises ``AssertionError`` when the callable disagrees with a closed form,
an invariant, a printed example or an independent library routine.  They run
against the real oracle (test_oracle_pins.py) and against deliberately broken
copies of it (test_oracle_mutants.py), which must each fail at least one pin.

Sources (page title, section):
  A = "第 11 章 · Attention 入门"
  S = "3.3 Self-Attention机制深入理解"
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

TIGHT = 1e-12


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def _qkv(B, Hq, Hkv, Tq, Tk, D, seed=0):
    return (_rand((B, Hq, Tq, D), seed), _rand((B, Hkv, Tk, D), seed + 1),
            _rand((B, Hkv, Tk, D), seed + 2))


def _expand_kv(x, Hq):
    """[B,Hkv,T,D] -> [B,Hq,T,D] with query head h reading kv head h//(Hq/Hkv)."""
    g = Hq // x.shape[1]
    return np.repeat(x, g, axis=1)


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def pin_causal_row0_returns_v0(attention):
    """S §10.2: row 0 sees only key 0, so its weight is 1 and o_0 = v_0;
    lse_0 is then the single scaled score s_00."""
    B, Hq, Hkv, T, D = 2, 4, 2, 9, 16
    q, k, v = _qkv(B, Hq, Hkv, T, T, D, seed=3)
    o, lse = attention(q, k, v, True)
    ve, ke = _expand_kv(v, Hq), _expand_kv(k, Hq)
    assert np.abs(o[:, :, 0, :] - ve[:, :, 0, :]).max() <= TIGHT
    s00 = (q[:, :, 0, :].astype(np.float64) * ke[:, :, 0, :]).sum(-1) / math.sqrt(D)
    assert np.abs(lse[:, :, 0] - s00).max() <= 1e-9


def pin_q_zero_gives_prefix_mean(attention):
    """Q = 0 makes every visible score 0, so the weights are uniform: the
    causal output is the running prefix mean of V (bottom-right aligned when
    Tq < Tk), the non-causal output is the column mean, and lse = ln(#visible)."""
    B, H, Tq, Tk, D = 1, 2, 5, 8, 4
    _, k, v = _qkv(B, H, H, Tq, Tk, D, seed=5)
    q = np.zeros((B, H, Tq, D), np.float32)
    o, lse = attention(q, k, v, True)
    vd = v.astype(np.float64)
    for i in range(Tq):
        n = i + (Tk - Tq) + 1
        assert np.abs(o[:, :, i, :] - vd[:, :, :n, :].mean(axis=2)).max() <= 1e-12
        assert np.abs(lse[:, :, i] - math.log(n)).max() <= 1e-12
    o, lse = attention(q, k, v, False)
    assert np.abs(o - vd.mean(axis=2, keepdims=True)).max() <= 1e-12
    assert np.abs(lse - math.log(Tk)).max() <= 1e-12


def pin_v_ones_gives_ones(attention):
    """S §3.4: each softmax row sums to 1, so V = 1 gives O = 1."""
    q, k, _ = _qkv(2, 3, 3, 7, 7, 8, seed=7)
    v = np.ones_like(k)
    for causal in (True, False):
        o, _ = attention(q, k, v, causal)
        assert np.abs(o - 1.0).max() <= 1e-12


def pin_two_keys_sigmoid(attention):
    """Two keys, hand-made vectors: q = (a, 0), k0 = (1, 0), k1 = (0, 1) and
    scale 1 give s0 = a, s1 = 0, so p0 = 1/(1 + e^-a) and lse = ln(e^a + 1)."""
    for a in (-3.0, 0.5, 2.0, 7.25):
        q = np.array([[[[a, 0.0]]]], np.float32)
        k = np.array([[[[1.0, 0.0], [0.0, 1.0]]]], np.float32)
        v = np.array([[[[2.0, -1.0], [-4.0, 0.5]]]], np.float32)
        o, lse = attention(q, k, v, False, scale=1.0)
        p0 = 1.0 / (1.0 + math.exp(-a))
        vd = v.astype(np.float64)
        want = p0 * vd[0, 0, 0] + (1 - p0) * vd[0, 0, 1]
        assert np.abs(o[0, 0, 0] - want).max() <= 1e-12
        assert abs(lse[0, 0, 0] - math.log(math.exp(a) + 1.0)) <= 1e-12


def pin_three_keys_causal_by_hand(attention):
    """T = 3 causal with q_i = (1, 0), k = rows (1,0), (2,0), (3,0), scale 1/2:
    s_ij = j'/2 with j' = j + 1.  Row 0 -> v0; row 1 -> weights
    (e^.5, e^1)/sum; row 2 -> (e^.5, e^1, e^1.5)/sum."""
    q = np.array([[[[1.0, 0.0]] * 3]], np.float32)
    k = np.array([[[[1.0, 0.0], [2.0, 0.0], [3.0, 0.0]]]], np.float32)
    v = np.array([[[[1.0, 10.0], [2.0, 20.0], [4.0, 40.0]]]], np.float32)
    o, lse = attention(q, k, v, True, scale=0.5)
    e = [math.exp(0.5), math.exp(1.0), math.exp(1.5)]
    rows = [[1.0, 0, 0], [e[0], e[1], 0], [e[0], e[1], e[2]]]
    for i, w in enumerate(rows):
        z = sum(w)
        want = sum(w[j] / z * v[0, 0, j].astype(np.float64) for j in range(3))
        assert np.abs(o[0, 0, i] - want).max() <= 1e-12
        assert abs(lse[0, 0, i] - math.log(z if i else e[0])) <= 1e-12


def pin_mask_matches_page_example(attention):
    """S §10.2 prints the 4x4 causal mask.  With V = identity the output row
    is the weight row P_i, so its support must be exactly the printed mask
    and every row must sum to 1 (weights of -inf entries are 0)."""
    mask = np.array([[int(x) for x in r] for r in read_golden("causal_mask_4x4.txt")])
    T = mask.shape[0]
    q, k, _ = _qkv(1, 1, 1, T, T, T, seed=11)
    v = np.eye(T, dtype=np.float32)[None, None]
    o, _ = attention(q, k, v, True)
    P = o[0, 0]
    assert np.array_equal(P > 0, mask == 1)
    assert np.abs(P.sum(-1) - 1.0).max() <= 1e-12


def pin_shape_trace(attention):
    """S §5.2 traces (1, 8, 6, 64) per-head tensors to (1, 8, 6, 6) weights and
    a (1, 8, 6, 64) context, dividing every score by sqrt(64) = 8."""
    g = {r[0]: [int(x) for x in r[1:]] for r in read_golden("shape_trace_t6.txt")}
    B, H, T, D = g["heads_q"]
    q, k, _ = _qkv(B, H, H, T, T, D, seed=13)
    # V = identity columns: context[..., :T] is the weight matrix itself.
    v = np.zeros((B, H, T, D), np.float32)
    v[..., :T] = np.eye(T, dtype=np.float32)
    o, lse = attention(q, k, v, False)
    assert list(o.shape) == g["context_heads"]
    w = o[..., :T]
    assert list(w.shape) == g["attn_weights"]
    assert np.abs(w.sum(-1) - 1.0).max() <= 1e-12
    # Explicit scale 1/8 must equal the default scale 1/sqrt(64).
    o8, lse8 = attention(q, k, v, False, scale=1.0 / g["scale_divisor"][0])
    assert np.abs(o8 - o).max() <= TIGHT and np.abs(lse8 - lse).max() <= TIGHT


def pin_lse_normalises_scores(attention):
    """sum_j exp(s_ij - lse_i) = 1 over the visible keys (definition of the
    row log-sum-exp of the scaled scores)."""
    B, Hq, Hkv, Tq, Tk, D = 1, 2, 1, 6, 9, 8
    q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=17)
    _, lse = attention(q, k, v, True)
    ke = _expand_kv(k, Hq).astype(np.float64)
    s = np.einsum("bhid,bhjd->bhij", q.astype(np.float64), ke) / math.sqrt(D)
    for i in range(Tq):
        n = i + Tk - Tq + 1
        tot = np.exp(s[:, :, i, :n] - lse[:, :, i, None]).sum(-1)
        assert np.abs(tot - 1.0).max() <= 1e-12


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------

def pin_permutations(attention):
    """Non-causal attention is equivariant in the query order and invariant to
    permuting the K and V rows together."""
    B, H, Tq, Tk, D = 2, 2, 7, 11, 8
    q, k, v = _qkv(B, H, H, Tq, Tk, D, seed=19)
    o, lse = attention(q, k, v, False)
    rng = np.random.default_rng(23)
    pq = rng.permutation(Tq)
    pk = rng.permutation(Tk)
    o2, lse2 = attention(q[:, :, pq], k, v, False)
    assert np.abs(o2 - o[:, :, pq]).max() <= 1e-12
    assert np.abs(lse2 - lse[:, :, pq]).max() <= 1e-12
    o3, lse3 = attention(q, k[:, :, pk], v[:, :, pk], False)
    assert np.abs(o3 - o).max() <= 1e-12
    assert np.abs(lse3 - lse).max() <= 1e-12


def pin_gqa_equals_repeated_mha(attention):
    """A §11.8.1 / S §9.3: GQA with group g equals MHA whose K/V heads are the
    shared head repeated g times; Hkv = 1 is MQA."""
    B, Hq, T, D = 1, 8, 6, 8
    for Hkv in (1, 2, 4):
        q, k, v = _qkv(B, Hq, Hkv, T, T, D, seed=29 + Hkv)
        for causal in (True, False):
            o, lse = attention(q, k, v, causal)
            o2, lse2 = attention(q, _expand_kv(k, Hq), _expand_kv(v, Hq), causal)
            assert np.abs(o - o2).max() <= TIGHT
            assert np.abs(lse - lse2).max() <= TIGHT


def pin_shift_invariance(attention):
    """S §7.2: softmax is unchanged by adding the same value to a whole row.
    Adding c to every K row adds scale * q_i . c to every score of row i, so O
    is unchanged and lse_i moves by exactly that amount."""
    B, H, T, D = 1, 2, 8, 8
    q, k, v = _qkv(B, H, H, T, T, D, seed=31)
    c = np.linspace(-2, 2, D).astype(np.float32)
    o, lse = attention(q, k, v, True)
    o2, lse2 = attention(q, k + c, v, True)
    shift = (q.astype(np.float64) * c.astype(np.float64)).sum(-1) / math.sqrt(D)
    assert np.abs(o2 - o).max() <= 1e-6  # k + c is rounded to float32
    assert np.abs(lse2 - (lse + shift)).max() <= 1e-5


def pin_large_scores_stay_finite(attention):
    """S §7.1/§7.2: with the row maximum subtracted, huge scores (Q x 100)
    cannot overflow: every output is finite and weights are convex."""
    q, k, v = _qkv(1, 2, 2, 16, 16, 64, seed=37)
    o, lse = attention(q * 100.0, k, v, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    vd = v.astype(np.float64)
    assert (o <= vd.max(axis=2, keepdims=True) + 1e-9).all()
    assert (o >= vd.min(axis=2, keepdims=True) - 1e-9).all()


def pin_block_merge_of_key_halves(attention):
    """S §12.3: two key blocks with their own (m, l, O) merge exactly into the
    full-row result.  With l = e^(lse - m) the page's formula reads
    lse = ln(e^lse1 + e^lse2), O = (e^lse1 O1 + e^lse2 O2) / e^lse."""
    B, Hq, Hkv, Tq, Tk, D = 1, 4, 2, 5, 12, 8
    q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=41)
    o, lse = attention(q, k, v, False)
    h = 5
    o1, l1 = attention(q, k[:, :, :h], v[:, :, :h], False)
    o2, l2 = attention(q, k[:, :, h:], v[:, :, h:], False)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    lse_m = m + np.log(w1 + w2)
    o_m = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    assert np.abs(lse_m - lse).max() <= 1e-12
    assert np.abs(o_m - o).max() <= 1e-12


def pin_rows_subset_matches_full(attention):
    """The row-sampling entry computes the same rows as the full call."""
    B, Hq, Hkv, Tq, Tk, D = 2, 4, 2, 9, 13, 16
    q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=43)
    o, lse = attention(q, k, v, True)
    rows = np.array([0, 5, 8, 17, 40, B * Hq * Tq - 1])
    o_r, lse_r = attention(q, k, v, True, rows=rows)
    assert np.abs(o_r - o.reshape(-1, D)[rows]).max() == 0.0
    assert np.abs(lse_r - lse.reshape(-1)[rows]).max() == 0.0


# --------------------------------------------------------------------------
# Independent routines
# --------------------------------------------------------------------------

def pin_torch_sdpa_f64(attention):
    """A §11 exercise 4 compares against torch's scaled_dot_product_attention;
    here it runs in float64 on the CPU with a bottom-right causal mask."""
    import torch
    import torch.nn.functional as F
    for (B, Hq, Hkv, Tq, Tk, D, causal) in [
            (1, 4, 4, 16, 16, 8, True), (2, 4, 2, 7, 19, 16, True),
            (1, 8, 1, 10, 10, 4, False), (1, 2, 2, 1, 33, 8, True)]:
        q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=47 + Tq)
        o, lse = attention(q, k, v, causal)
        tq = torch.from_numpy(q).double()
        tk = torch.from_numpy(_expand_kv(k, Hq)).double()
        tv = torch.from_numpy(_expand_kv(v, Hq)).double()
        mask = None
        if causal:
            i = torch.arange(Tq)[:, None]
            j = torch.arange(Tk)[None, :]
            mask = j <= i + (Tk - Tq)
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
        assert np.abs(o - ref.numpy()).max() <= 1e-12
        s = torch.einsum("bhid,bhjd->bhij", tq, tk) / math.sqrt(D)
        if mask is not None:
            s = s.masked_fill(~mask, float("-inf"))
        assert np.abs(lse - torch.logsumexp(s, -1).numpy()).max() <= 1e-12


def pin_brute_force_tiny(attention):
    """Literal definition on tiny inputs with Python floats: weights
    exp(s_ij) / sum exp(s_ij) over the visible keys (no max subtraction)."""
    B, Hq, Hkv, Tq, Tk, D = 1, 2, 1, 4, 6, 3
    q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=53)
    for causal in (True, False):
        o, lse = attention(q, k, v, causal)
        for h in range(Hq):
            for i in range(Tq):
                vis = [j for j in range(Tk) if (not causal) or j <= i + Tk - Tq]
                sc = {j: sum(float(q[0, h, i, d]) * float(k[0, 0, j, d])
                             for d in range(D)) / math.sqrt(D) for j in vis}
                z = sum(math.exp(sc[j]) for j in vis)
                for d in range(D):
                    want = sum(math.exp(sc[j]) / z * float(v[0, 0, j, d]) for j in vis)
                    assert abs(o[0, h, i, d] - want) <= 1e-12
                assert abs(lse[0, h, i] - math.log(z)) <= 1e-12


def pin_window_brute_force_tiny(attention):
    """Sliding window ("第 11 章 · Attention 入门" §11.8.4: only the most recent
    W tokens), literal definition on tiny inputs: row i sees keys
    i + Tk - Tq - W + 1 .. i + Tk - Tq (Tq < Tk, so the offset matters)."""
    B, Hq, Hkv, Tq, Tk, D = 1, 2, 1, 4, 7, 3
    q, k, v = _qkv(B, Hq, Hkv, Tq, Tk, D, seed=54)
    for W in (1, 2, 3, 5):
        o, lse = attention(q, k, v, True, window=W)
        for h in range(Hq):
            for i in range(Tq):
                a = i + Tk - Tq
                vis = [j for j in range(Tk) if a - W < j <= a]
                sc = {j: sum(float(q[0, h, i, d]) * float(k[0, 0, j, d])
                             for d in range(D)) / math.sqrt(D) for j in vis}
                z = sum(math.exp(sc[j]) for j in vis)
                for d in range(D):
                    want = sum(math.exp(sc[j]) / z * float(v[0, 0, j, d]) for j in vis)
                    assert abs(o[0, h, i, d] - want) <= 1e-12
                assert abs(lse[0, h, i] - math.log(z)) <= 1e-12


def pin_window_of_one_returns_own_value(attention):
    """W = 1: each row sees only the key at its own position, so O_i is that
    key's value row and lse_i its scaled score."""
    q, k, v = _qkv(2, 4, 2, 5, 9, 8, seed=55)
    o, lse = attention(q, k, v, True, window=1)
    kx, vx = _expand_kv(k, 4), _expand_kv(v, 4)
    for i in range(5):
        j = i + 4
        assert np.array_equal(o[:, :, i], vx[:, :, j].astype(np.float64))
        s = (q[:, :, i].astype(np.float64) * kx[:, :, j].astype(np.float64)).sum(-1) / math.sqrt(8)
        assert np.abs(lse[:, :, i] - s).max() <= 1e-12


def pin_window_covering_every_key_is_causal(attention):
    q, k, v = _qkv(1, 2, 2, 6, 10, 4, seed=56)
    o, lse = attention(q, k, v, True)
    for W in (10, 11, 1000):
        o2, lse2 = attention(q, k, v, True, window=W)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def pin_window_q_zero_gives_window_mean(attention):
    """Q = 0: equal weights over the window, O_i = mean of its value rows,
    lse_i = ln(number of keys in the window)."""
    _, k, v = _qkv(1, 2, 1, 6, 11, 4, seed=57)
    q = np.zeros((1, 2, 6, 4), np.float32)
    W = 4
    o, lse = attention(q, k, v, True, window=W)
    for i in range(6):
        a = i + 5
        j0 = max(0, a - W + 1)
        want = v[0, 0, j0:a + 1].astype(np.float64).mean(0)
        assert np.abs(o[0, :, i] - want).max() <= 1e-12
        assert np.abs(lse[0, :, i] - math.log(a + 1 - j0)).max() <= 1e-12


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
