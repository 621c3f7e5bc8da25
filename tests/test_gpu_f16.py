"""fp16 I/O ("第 11 章 · Attention 入门" §11.8.5: 16-bit inputs and outputs
with fp32 accumulation) on the tensor-core prefill and the stream-K decode,
against the float64 oracle on the same fp16-rounded inputs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, sample_rows, to_dev
from transformer_attention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

# fp16 keeps 11 significant bits against bf16's 8; the 16-bit tolerances of
# the bf16 path apply unchanged.
TOL_O_F16, TOL_LSE_F16 = TOL_O_BF16, TOL_LSE_BF16


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,D", [
    (1, 4, 4, 128, 128, 64), (2, 8, 2, 300, 300, 128), (1, 6, 3, 257, 700, 64),
    (1, 8, 1, 1000, 1000, 128),
])
@pytest.mark.parametrize("causal", [True, False])
def test_f16_prefill_matches_oracle(B, Hq, Hkv, Tq, Tk, D, causal):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, D, "f16", seed=101)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_F16, TOL_LSE_F16, f"f16 prefill {B,Hq,Hkv,Tq,Tk,D}")


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (16, 16, 64), (32, 1, 128), (64, 8, 64)])
def test_f16_decode_matches_oracle(Hq, Hkv, D):
    a = attn()
    q, k, v = make_qkv(4, Hq, Hkv, 1, 1500, D, "f16", seed=102)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=False)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_F16, TOL_LSE_F16, f"f16 decode Hq{Hq} Hkv{Hkv}")


def test_f16_window_matches_oracle():
    a = attn()
    q, k, v = make_qkv(1, 8, 2, 700, 900, 128, "f16", seed=103)
    o, lse = a.attn_fwd_window(*to_dev(q, k, v), 300)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, True, window=300)
    compare(o, lse, o_ref, lse_ref, TOL_O_F16, TOL_LSE_F16, "f16 window 300")


@pytest.mark.parametrize("causal", [True, False])
def test_f16_rising_scores_stay_finite(causal):
    """Scores rising along the key axis far faster than fp16's range (2^16):
    weights against a stale reference would overflow fp16 P, so the fast path
    must hand such tiles to the exact path."""
    a = attn()
    g = torch.Generator().manual_seed(104)
    T, D = 512, 64
    ramp = torch.linspace(0.0, 6.0, T)[None, None, :, None]
    q = (torch.ones(1, 2, T, D) + 0.3 * torch.randn(1, 2, T, D, generator=g)).half()
    k = (ramp + 0.5 * torch.randn(1, 2, T, D, generator=g)).half()
    v = torch.randn(1, 2, T, D, generator=g).half()
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_F16, 1e-3 * max(1.0, float(abs(lse_ref).max())) / 10)


def test_f16_full_size_sampled():
    """Llama-3-8B shapes at T = 8192 in fp16, sampled rows."""
    a = attn()
    B, Hq, Hkv, T, D = 1, 32, 8, 8192, 128
    q, k, v = make_qkv(B, Hq, Hkv, T, T, D, "f16", seed=105)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=True)
    check_status(a)
    rows = sample_rows(B, Hq, T, 1500, seed=6)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, True, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    compare(o.reshape(-1, D)[idx], lse.reshape(-1)[idx], o_ref, lse_ref, TOL_O_F16, TOL_LSE_F16,
            "f16 T8192")


def test_f16_is_more_precise_than_bf16():
    """The same values in both 16-bit formats (drawn in bf16, with the
    entries below 2^-12 set to 0 so that fp16 holds every value exactly):
    fp16's finer P and O rounding must not be worse than bf16's."""
    a = attn()
    qb, kb, vb = (torch.where(x.float().abs() < 2.0 ** -12, 0.0, x.float()).to(torch.bfloat16)
                  for x in make_qkv(1, 8, 8, 512, 512, 128, "bf16", seed=106))
    qh, kh, vh = qb.half(), kb.half(), vb.half()
    for xb, xh in ((qb, qh), (kb, kh), (vb, vh)):
        assert torch.equal(xh.float(), xb.float())
    o_ref, _ = oracle.attention_f64(qb, kb, vb, True)
    ob, _ = a.attn_fwd(*to_dev(qb, kb, vb), causal=True)
    oh, _ = a.attn_fwd(*to_dev(qh, kh, vh), causal=True)
    check_status(a)
    eb = np.abs(ob.float().cpu().numpy() - o_ref).max()
    eh = np.abs(oh.float().cpu().numpy() - o_ref).max()
    assert eh <= eb, (eh, eb)


@pytest.mark.parametrize("causal", [True, False])
def test_f16_varlen_matches_oracle(causal):
    from transformer_attention_fwd_gb300.inputs import make_varlen
    a = attn()
    lq, lk = [1, 127, 300, 0, 700], [1, 127, 600, 5, 700]
    if not causal:
        lk = lq[:3] + [5, 700]
    q, k, v, cq, ck = make_varlen(lq, lk, 8, 2, 128, seed=107, dtype="f16")
    o, lse = a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), causal)
    check_status(a)
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, causal)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= TOL_O_F16
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= TOL_LSE_F16


def test_f16_paged_decode_matches_oracle():
    from transformer_attention_fwd_gb300.inputs import make_paged
    a = attn()
    q, kv, bt, sl = make_paged(5, 16, 4, 128, 16, [1000, 1, 0, 77, 2048], seed=108, dtype="f16")
    o, lse = a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    check_status(a)
    assert o.dtype == torch.float16
    o_ref, lse_ref = oracle.decode_paged_f64(q, kv, bt, sl)
    o_g = o.float().cpu().numpy()[:, :, 0, :]
    assert np.abs(o_g - o_ref).max() <= TOL_O_F16
    l_g, fin = lse.cpu().numpy(), np.isfinite(lse_ref)
    assert (np.isfinite(l_g) == fin).all() and np.abs(l_g[fin] - lse_ref[fin]).max() <= TOL_LSE_F16
