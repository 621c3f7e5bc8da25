"""The paged-cache decode oracle against cases written out by hand and
against properties that pin the token -> (block, row) map ("第 11 章 ·
Attention 入门", 11.11, the KV-cache / VMM passage: block_table[req][t/16]
names the physical block of token t)."""
import math

import numpy as np
import pytest

import oracle


def _softmax_weighted(q, keys, vals, scale):
    """Plain softmax(q.k * scale) . v for one head, written out."""
    s = [scale * sum(float(qi) * float(ki) for qi, ki in zip(q, k)) for k in keys]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    o = [sum(wj * v[d] for wj, v in zip(w, vals)) / z for d in range(len(q))]
    return o, m + math.log(z)


def pin_hand_built_block_table(fn=oracle.decode_paged_f64):
    # page_size 2, one KV head, D = 2, five blocks.  Request 0 has 3 keys in
    # blocks [3, 1] (t=0,1 -> block 3 rows 0,1; t=2 -> block 1 row 0);
    # request 1 has 1 key in block 4 row 0.  Everything else is NaN.
    kv = np.full((5, 2, 1, 2, 2), np.nan, np.float32)
    kv[3, 0, 0, 0] = [1.0, 0.0]; kv[3, 1, 0, 0] = [10.0, 1.0]
    kv[3, 0, 0, 1] = [0.0, 1.0]; kv[3, 1, 0, 1] = [20.0, 2.0]
    kv[1, 0, 0, 0] = [1.0, 1.0]; kv[1, 1, 0, 0] = [30.0, 3.0]
    kv[4, 0, 0, 0] = [-1.0, 2.0]; kv[4, 1, 0, 0] = [5.0, 6.0]
    bt = np.array([[3, 1, 0], [4, 2, 2]])
    sl = np.array([3, 1])
    q = np.array([[[0.5, -1.0], [2.0, 1.0]], [[1.0, 1.0], [0.0, 3.0]]], np.float32)  # [B, Hq=2, D]
    o, lse = fn(q, kv, bt, sl, scale=0.7)
    keys0 = [[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]
    vals0 = [[10.0, 1.0], [20.0, 2.0], [30.0, 3.0]]
    for h in range(2):
        want_o, want_l = _softmax_weighted(q[0, h], keys0, vals0, 0.7)
        assert np.allclose(o[0, h], want_o, rtol=0, atol=1e-12)
        assert abs(lse[0, h] - want_l) < 1e-12
        want_o, want_l = _softmax_weighted(q[1, h], [[-1.0, 2.0]], [[5.0, 6.0]], 0.7)
        assert np.allclose(o[1, h], want_o, rtol=0, atol=1e-12)
        assert abs(lse[1, h] - want_l) < 1e-12


def pin_empty_request_gives_zero_output_and_minus_inf_lse(fn=oracle.decode_paged_f64):
    kv = np.ones((2, 2, 1, 4, 8), np.float32)
    o, lse = fn(np.ones((2, 2, 8), np.float32), kv, np.zeros((2, 1), np.int64),
                np.array([0, 4]))
    assert (o[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.allclose(o[1], 1.0) and np.allclose(lse[1], math.log(4) + 8 / math.sqrt(8))


def pin_contiguous_pages_equal_dense_cache(fn=oracle.decode_paged_f64):
    """Blocks laid out in token order hold exactly the dense cache: the paged
    result equals the dense oracle on the dense tensors (GQA, ragged last
    page)."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, P, L = 2, 4, 2, 16, 4, 11
    kd = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    vd = rng.standard_normal((B, Hkv, L, D)).astype(np.float32)
    npg = -(-L // P)
    kv = np.zeros((B * npg, 2, Hkv, P, D), np.float32)
    for b in range(B):
        for t in range(L):
            kv[b * npg + t // P, 0, :, t % P] = kd[b, :, t]
            kv[b * npg + t // P, 1, :, t % P] = vd[b, :, t]
    bt = np.arange(B * npg).reshape(B, npg)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    o, lse = fn(q, kv, bt, np.array([L, L]))
    od, ld = oracle.attention_f64(q[:, :, None, :], kd, vd, False)
    assert np.array_equal(o, od[:, :, 0]) and np.array_equal(lse, ld[:, :, 0])


def pin_block_permutation_and_unused_rows_do_not_matter(fn=oracle.decode_paged_f64):
    """Moving blocks to other physical ids (and updating the table) changes
    nothing; NaN in rows past the sequence end or in unreferenced blocks is
    never read."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, P = 3, 2, 1, 8, 4
    lens = np.array([1, 9, 12])
    nb = 12
    kv = rng.standard_normal((nb, 2, Hkv, P, D)).astype(np.float32)
    bt = rng.permutation(nb)[:9].reshape(B, 3)
    for b in range(B):  # poison rows past each sequence end
        for t in range(lens[b], 3 * P):
            kv[bt[b, t // P], :, :, t % P] = np.nan
    used = set(bt[b, t // P] for b in range(B) for t in range(lens[b]))
    for blk in range(nb):
        if blk not in used and blk not in bt:
            kv[blk] = np.nan
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    o, lse = fn(q, kv, bt, lens)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    perm = rng.permutation(nb)
    kv2 = np.empty_like(kv)
    kv2[perm] = kv
    o2, lse2 = fn(q, kv2, perm[bt], lens)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_rejects_bad_tables():
    kv = np.zeros((2, 2, 1, 4, 8), np.float32)
    q = np.zeros((1, 1, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.decode_paged_f64(q, kv, np.array([[5]]), np.array([3]))  # block id out of range
    with pytest.raises(ValueError):
        oracle.decode_paged_f64(q, kv, np.array([[0]]), np.array([5]))  # longer than the table


PINS = [pin_hand_built_block_table, pin_empty_request_gives_zero_output_and_minus_inf_lse,
        pin_contiguous_pages_equal_dense_cache, pin_block_permutation_and_unused_rows_do_not_matter]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_paged_oracle_pin(pin):
    pin()


# Plausible mistakes planted in a copy of the gather (on the CPU; the real
# oracle is never modified).  Each must fail at least one pin.
MUTANTS = [
    ("row_from_page_index", "k = kv[blk, 0, :, t % P, :]", "k = kv[blk, 0, :, t // P, :]"),
    ("k_and_v_swapped", "k = kv[blk, 0, :, t % P, :]", "k = kv[blk, 1, :, t % P, :]"),
    ("table_row_of_request_0", "blk = bt[b, t // P]", "blk = bt[0, t // P]"),
    ("page_from_row_index", "blk = bt[b, t // P]", "blk = bt[b, t % P]"),
    ("last_key_dropped", "t = np.arange(L)", "t = np.arange(max(L - 1, 1))"),
    ("heads_not_moved_first", "k = np.ascontiguousarray(k.transpose(1, 0, 2))[None]",
     "k = np.ascontiguousarray(k.reshape(k.shape[1], k.shape[0], k.shape[2]))[None]"),
    ("empty_request_lse_zero", "lse = np.full((B, Hq), -np.inf, dtype=np.float64)",
     "lse = np.zeros((B, Hq), dtype=np.float64)"),
]


def _mutant(old, new):
    import inspect
    import textwrap
    src = textwrap.dedent(inspect.getsource(oracle.decode_paged_f64))
    assert old in src, old
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new, 1), "<mutant>", "exec"), ns)
    return ns["decode_paged_f64"]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_paged_mutant_is_caught(name, old, new):
    fn = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(fn)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches {name}"
