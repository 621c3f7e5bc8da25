"""Packed variable-length prefill against the float64 oracle: sequences back
to back along the token axis of (T, H, D) tensors ("第 11 章 · Attention
入门", 11.11), each its own attention problem (bottom-right causal for a
query chunk against a longer history, §11.8.2; sliding window, §11.8.4)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status
from transformer_attention_fwd_gb300.inputs import VARLEN_WORKLOADS, make_varlen, make_varlen_workload

pytestmark = pytest.mark.gpu


def _run(a, q, k, v, cq, ck, causal, window=0):
    o, lse = a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), causal,
                               window=window)
    check_status(a)
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _compare(o, lse, o_ref, lse_ref, rows, what):
    """Rows (token indices) of o [total_q, Hq, D] and lse [Hq, total_q]."""
    err_o = np.abs(o[rows] - o_ref[rows]).max() if len(rows) else 0.0
    lr, lg = lse_ref[:, rows], lse[:, rows]
    fin = np.isfinite(lr)
    assert (np.isfinite(lg) == fin).all(), f"{what}: lse finiteness differs"
    assert (lg[~fin] == lr[~fin]).all(), f"{what}: non-finite lse differs"
    err_l = np.abs(lg[fin] - lr[fin]).max() if fin.any() else 0.0
    assert err_o <= TOL_O_BF16, f"{what}: max |O - O_ref| = {err_o:.3e}"
    assert err_l <= TOL_LSE_BF16, f"{what}: max |lse - lse_ref| = {err_l:.3e}"


MIXES = {
    # tile edges, one-row sequences and an empty one, all in one launch
    "edges": ([1, 127, 128, 129, 255, 256, 257, 0, 700, 3], None),
    # query chunks against longer histories (chunked prefill)
    "chunks": ([64, 300, 1, 129, 256], [1000, 300, 517, 900, 256]),
    "long_short": ([2000, 5, 1100, 37], None),
}


@pytest.mark.parametrize("mix", list(MIXES))
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_matches_oracle(mix, D, causal):
    a = attn()
    lq, lk = MIXES[mix]
    lk = lq if lk is None else lk
    q, k, v, cq, ck = make_varlen(lq, lk, 8, 2, D, seed=81)
    o, lse = _run(a, q, k, v, cq, ck, causal)
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, causal)
    _compare(o, lse, o_ref, lse_ref, np.arange(q.shape[0]), f"{mix} D{D} causal={causal}")


@pytest.mark.parametrize("window", [1, 100, 128, 300])
def test_varlen_window_matches_oracle(window):
    a = attn()
    lq, lk = [700, 1, 300, 129], [700, 40, 1000, 129]
    q, k, v, cq, ck = make_varlen(lq, lk, 4, 4, 128, seed=82)
    o, lse = _run(a, q, k, v, cq, ck, True, window)
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, True, window=window)
    _compare(o, lse, o_ref, lse_ref, np.arange(q.shape[0]), f"window {window}")


def test_equal_lengths_equal_the_dense_kernel_exactly():
    """B sequences of one length, packed, give the dense [B, H, T, D] result
    bit for bit: the same tiles, and keys of the neighbouring sequence get an
    exact zero weight where the dense tensor has zero fill."""
    a = attn()
    B, Hq, Hkv, T, D = 3, 8, 2, 700, 128
    q, k, v, cq, ck = make_varlen([T] * B, [T] * B, Hq, Hkv, D, seed=83)
    for causal in (True, False):
        o, lse = a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), causal)
        qd = q.view(B, T, Hq, D).transpose(1, 2).contiguous().cuda()
        kd = k.view(B, T, Hkv, D).transpose(1, 2).contiguous().cuda()
        vd = v.view(B, T, Hkv, D).transpose(1, 2).contiguous().cuda()
        od, ld = a.attn_fwd_prefill(qd, kd, vd, causal=causal)
        check_status(a)
        assert torch.equal(o.view(B, T, Hq, D).transpose(1, 2), od)
        assert torch.equal(lse.view(Hq, B, T).transpose(0, 1), ld)


def test_sequence_without_keys_gets_zero_and_minus_inf():
    a = attn()
    q, k, v, cq, ck = make_varlen([5, 3, 4], [0, 6, 0], 4, 2, 64, seed=84)
    o, lse = _run(a, q, k, v, cq, ck, False)
    assert (o[:5] == 0).all() and (o[8:] == 0).all()
    assert np.isneginf(lse[:, :5]).all() and np.isneginf(lse[:, 8:]).all()
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, False)
    _compare(o, lse, o_ref, lse_ref, np.arange(5, 8), "middle sequence")


def test_bad_offsets_are_reported_and_skipped():
    a = attn()
    q, k, v, _, ck = make_varlen([100, 50], [100, 50], 4, 4, 64, seed=85)
    # Sequence 0 then has 120 query rows against 100 keys, which the causal
    # alignment cannot place: it is dropped; sequence 1 is still computed.
    bad_q = torch.tensor([0, 120, 150], dtype=torch.int32)
    o = torch.full((150, 4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((4, 150), 7.0, dtype=torch.float32, device="cuda")
    a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), bad_q.cuda(), ck.cuda(), True, out=o, lse=lse)
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    assert (o[:120] == 7.0).all() and (lse[:, :120] == 7.0).all()
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, bad_q, ck, True, seqs=[1])
    _compare(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, np.arange(120, 150),
             "sequence after a dropped one")
    # An offset past the end of q.
    out_of_range = torch.tensor([0, 100, 400], dtype=torch.int32)
    a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), out_of_range.cuda(), ck.cuda(), False)
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    # Decreasing key offsets.
    a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.tensor([0, 100, 150], dtype=torch.int32).cuda(),
                      torch.tensor([0, 120, 100], dtype=torch.int32).cuda(), False)
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    check_status(a)


def test_no_query_rows_launches_nothing():
    a = attn()
    q = torch.empty((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((10, 4, 64), dtype=torch.bfloat16, device="cuda")
    cq = torch.zeros(3, dtype=torch.int32, device="cuda")
    ck = torch.tensor([0, 4, 10], dtype=torch.int32, device="cuda")
    o, lse = a.attn_fwd_varlen(q, k, k, cq, ck, True)
    check_status(a)
    assert o.shape == (0, 4, 64) and a.last_launch_info()[2] == 0


def test_full_size_mix_sampled():
    """The packed Llama-3-8B workload of the bench (32 sequences of 128 to
    8192 tokens): every row of five sequences, including the longest and the
    shortest, against the oracle."""
    w = next(iter(VARLEN_WORKLOADS.values()))
    a = attn()
    q, k, v, cq, ck = make_varlen_workload(w, seed=0)
    o, lse = _run(a, q, k, v, cq, ck, w.causal)
    L = np.array(w.seqlens())
    pick = sorted({int(L.argmax()), int(L.argmin()), 2, 9, 17})
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, w.causal, seqs=pick)
    c = cq.numpy()
    rows = np.concatenate([np.arange(c[b], c[b + 1]) for b in pick])
    _compare(o, lse, o_ref, lse_ref, rows, "packed Llama-3 mix")
