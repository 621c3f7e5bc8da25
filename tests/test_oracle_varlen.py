"""The packed variable-length oracle against brute force and closed forms
that pin the sequence -> rows map ("第 11 章 · Attention 入门", 11.11, the
(T, H, D) layout; §11.8.2 for the bottom-right causal alignment of a query
chunk against a longer key history; §11.8.4 for the window)."""
import math

import numpy as np
import pytest

import oracle


def _brute(q, k, v, cq, ck, causal, scale, window=0):
    """Pure-Python loops: every (sequence, head, row) written out."""
    TQ, Hq, D = q.shape
    Hkv = k.shape[1]
    o = np.zeros((TQ, Hq, D))
    lse = np.full((Hq, TQ), np.nan)
    for b in range(len(cq) - 1):
        Tq, Tk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            for i in range(Tq):
                last = i + Tk - Tq if causal else Tk - 1
                first = max(0, last - window + 1) if window > 0 else 0
                keys = range(first, last + 1)
                if len(keys) == 0:
                    lse[h, cq[b] + i] = -math.inf
                    continue
                s = [scale * sum(float(q[cq[b] + i, h, d]) * float(k[ck[b] + j, hk, d])
                                 for d in range(D)) for j in keys]
                m = max(s)
                w = [math.exp(x - m) for x in s]
                z = sum(w)
                for d in range(D):
                    o[cq[b] + i, h, d] = sum(wj * float(v[ck[b] + j, hk, d])
                                             for wj, j in zip(w, keys)) / z
                lse[h, cq[b] + i] = m + math.log(z)
    return o, lse


def _rand(TQ, TK, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((TQ, Hq, D)).astype(np.float32),
            rng.standard_normal((TK, Hkv, D)).astype(np.float32),
            rng.standard_normal((TK, Hkv, D)).astype(np.float32))


def pin_brute_force(fn=oracle.attention_varlen_f64):
    # Three sequences (one without queries), GQA 4:2, chunk rows shorter than
    # their key history.
    cq, ck = [0, 3, 3, 8], [0, 4, 6, 11]
    q, k, v = _rand(8, 11, 4, 2, 3, seed=1)
    for causal in (False, True):
        for window in ((0, 2) if causal else (0,)):
            o, lse = fn(q, k, v, np.array(cq), np.array(ck), causal, 0.6, window=window)
            o_w, l_w = _brute(q, k, v, cq, ck, causal, 0.6, window)
            assert np.allclose(o, o_w, rtol=0, atol=1e-12)
            assert np.allclose(lse[:, :8], l_w[:, :8], rtol=0, atol=1e-12, equal_nan=True)


def pin_constant_values_and_zero_queries(fn=oracle.attention_varlen_f64):
    """V = c(b, h) on every key of sequence b, head h: each output row is
    c(b, h) (to float64 rounding).  Q = 0: every visible key weighs the same, so lse is
    ln(number of visible keys): min(Tk, i + Tk - Tq + 1) under the causal
    mask, capped at W with a window."""
    cq = np.array([0, 5, 5, 9, 16])
    ck = np.array([0, 7, 9, 13, 22])
    Hq, Hkv, D = 4, 2, 8
    rng = np.random.default_rng(2)
    q = np.zeros((16, Hq, D), np.float32)
    k = rng.standard_normal((22, Hkv, D)).astype(np.float32)
    v = np.zeros((22, Hkv, D), np.float32)
    for b in range(4):
        for hk in range(Hkv):
            v[ck[b]:ck[b + 1], hk, :] = 1.0 + b + 10.0 * hk
    for causal, window in ((False, 0), (True, 0), (True, 3)):
        o, lse = fn(q, k, v, cq, ck, causal, 0.5, window=window)
        for b in range(4):
            Tq, Tk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
            for i in range(Tq):
                n = min(Tk, i + Tk - Tq + 1) if causal else Tk
                if window:
                    n = min(n, window)
                for h in range(Hq):
                    assert np.allclose(o[cq[b] + i, h], 1.0 + b + 10.0 * (h // 2),
                                       rtol=1e-14, atol=0)
                    assert abs(lse[h, cq[b] + i] - math.log(n)) < 1e-14


def pin_sequences_without_keys(fn=oracle.attention_varlen_f64):
    cq, ck = np.array([0, 2, 5]), np.array([0, 0, 3])
    q, k, v = _rand(5, 3, 2, 2, 4, seed=3)
    o, lse = fn(q, k, v, cq, ck, False)
    assert (o[:2] == 0).all() and np.isneginf(lse[:, :2]).all()
    assert np.isfinite(lse[:, 2:]).all() and (o[2:] != 0).any()


def pin_packing_order_does_not_matter(fn=oracle.attention_varlen_f64):
    """The same sequences packed in reverse order give the same rows."""
    tq, tk = [4, 1, 6], [9, 3, 6]
    Hq, Hkv, D = 2, 1, 5
    seqs = [_rand(a, b, Hq, Hkv, D, seed=10 + i) for i, (a, b) in enumerate(zip(tq, tk))]

    def pack(order):
        q = np.concatenate([seqs[i][0] for i in order])
        k = np.concatenate([seqs[i][1] for i in order])
        v = np.concatenate([seqs[i][2] for i in order])
        cq = np.concatenate([[0], np.cumsum([tq[i] for i in order])])
        ck = np.concatenate([[0], np.cumsum([tk[i] for i in order])])
        return q, k, v, cq, ck

    fwd = fn(*pack([0, 1, 2]), True)
    rev = fn(*pack([2, 1, 0]), True)
    cq_f = np.concatenate([[0], np.cumsum(tq)])
    cq_r = np.concatenate([[0], np.cumsum(tq[::-1])])
    for i in range(3):
        r = 2 - i
        assert np.array_equal(fwd[0][cq_f[i]:cq_f[i + 1]], rev[0][cq_r[r]:cq_r[r + 1]])
        assert np.array_equal(fwd[1][:, cq_f[i]:cq_f[i + 1]], rev[1][:, cq_r[r]:cq_r[r + 1]])


def test_rejects_bad_offsets():
    q, k, v = _rand(4, 4, 1, 1, 2, seed=4)
    with pytest.raises(ValueError):
        oracle.attention_varlen_f64(q, k, v, np.array([0, 3, 2]), np.array([0, 2, 4]), False)
    with pytest.raises(ValueError):
        oracle.attention_varlen_f64(q, k, v, np.array([0, 5]), np.array([0, 4]), False)
    with pytest.raises(ValueError):  # causal chunk with more queries than keys
        oracle.attention_varlen_f64(q, k, v, np.array([0, 4]), np.array([0, 3]), True)


PINS = [pin_brute_force, pin_constant_values_and_zero_queries, pin_sequences_without_keys,
        pin_packing_order_does_not_matter]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_varlen_oracle_pin(pin):
    pin()


# Plausible mistakes planted in a copy of the slicing (on the CPU; the real
# oracle is never modified).  Each must fail at least one pin.
MUTANTS = [
    ("key_rows_from_query_offsets",
     "q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])",
     "q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(cq[b]), int(cq[b + 1])"),
    ("heads_not_moved_first",
     "qb = np.ascontiguousarray(q[q0:q1].transpose(1, 0, 2))[None]",
     "qb = np.ascontiguousarray(q[q0:q1].reshape(Hq, q1 - q0, D))[None]"),
    ("values_from_keys", "vb = np.ascontiguousarray(v[k0:k1]", "vb = np.ascontiguousarray(k[k0:k1]"),
    ("output_not_moved_back", "o[q0:q1] = ob[0].transpose(1, 0, 2)",
     "o[q0:q1] = ob[0].reshape(q1 - q0, Hq, D)"),
    ("empty_keys_lse_zero", "lse[:, q0:q1] = -np.inf", "lse[:, q0:q1] = 0.0"),
    ("causal_dropped", "attention_f64(qb, kb, vb, causal,", "attention_f64(qb, kb, vb, False,"),
    ("window_dropped", "None, nthreads, window)", "None, nthreads, 0)"),
    ("last_sequence_skipped", "for b in (range(B) if", "for b in (range(B - 1) if"),
]


def _mutant(old, new):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.attention_varlen_f64))
    assert old in src, old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new, 1), "<mutant>", "exec"), ns)
    return ns["attention_varlen_f64"]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_varlen_mutant_is_caught(name, old, new):
    fn = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(fn)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches {name}"
