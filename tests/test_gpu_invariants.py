"""Closed forms and invariants checked on the CUDA kernels themselves
("3.3 Self-Attention机制深入理解" §3.4 rows sum to 1, §7.2 shift invariance,
§9.3 GQA/MHA, §10.2 masked weights are 0; "第 11 章 · Attention 入门" §11.8.1).

Where each output row is computed independently with the same arithmetic
(causal row 0, V = 1, query permutation, GQA vs repeated MHA) the check is
bit-exact; elsewhere it uses the parity tolerances."""
import math

import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, TOL_O_F32, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def _run(a, q, k, v, causal, dtype):
    if dtype == "bf16" and q.shape[2] == 1 and not causal:
        return a.attn_fwd_decode(q, k, v)
    return a.attn_fwd(q, k, v, causal=causal)


@pytest.mark.parametrize("D", [64, 128])
def test_causal_row0_is_v0_exactly(D):
    a = attn()
    q, k, v = to_dev(*make_qkv(2, 4, 2, 300, 300, D, "bf16", seed=61))
    o, lse = a.attn_fwd(q, k, v, causal=True)
    check_status(a)
    ve = v.repeat_interleave(2, dim=1)
    assert torch.equal(o[:, :, 0, :], ve[:, :, 0, :])
    ke = k.repeat_interleave(2, dim=1)
    s00 = (q[:, :, 0, :].double() * ke[:, :, 0, :].double()).sum(-1) / math.sqrt(D)
    assert (lse[:, :, 0].double() - s00).abs().max().item() <= 1e-4


@pytest.mark.parametrize("dtype,causal,Tq,Tk", [("bf16", True, 300, 300), ("bf16", False, 200, 333),
                                                ("bf16", True, 130, 500), ("bf16", False, 1, 999),
                                                ("f32", True, 70, 70)])
def test_v_ones_gives_ones_exactly(dtype, causal, Tq, Tk):
    a = attn()
    q, k, _ = make_qkv(1, 4, 2, Tq, Tk, 128, dtype, seed=62)
    v = torch.ones_like(k)
    q, k, v = to_dev(q, k, v)
    o, _ = _run(a, q, k, v, causal, dtype)
    check_status(a)
    if dtype == "bf16":
        assert torch.equal(o, torch.ones_like(o))
    else:
        assert (o - 1).abs().max().item() <= TOL_O_F32


@pytest.mark.parametrize("causal", [True, False])
def test_q_zero_gives_prefix_mean(causal):
    a = attn()
    _, k, v = make_qkv(1, 2, 1, 200, 260, 64, "bf16", seed=63)
    q = torch.zeros(1, 2, 200, 64, dtype=torch.bfloat16)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    vd = v.double()[0, 0]
    off = 260 - 200
    for i in (0, 1, 57, 128, 199):
        n = i + off + 1 if causal else 260
        want = vd[:n].mean(0)
        assert (o[0, :, i].double().cpu() - want).abs().max().item() <= TOL_O_BF16
        assert (lse[0, :, i].double().cpu() - math.log(n)).abs().max().item() <= TOL_LSE_BF16


def test_identity_v_extracts_weights_with_exact_zero_mask():
    """V = identity (Tk = D = 128): O's row i is the weight row P_i.  Masked
    (future) keys must get weight exactly 0 and every row sums to 1."""
    a = attn()
    T = 128
    q, k, _ = make_qkv(1, 2, 2, T, T, 128, "bf16", seed=64)
    v = torch.eye(T, dtype=torch.bfloat16).expand(1, 2, T, T).contiguous()
    o, _ = a.attn_fwd(*to_dev(q, k, v), causal=True)
    check_status(a)
    P = o.float().cpu()
    upper = torch.triu(torch.ones(T, T, dtype=torch.bool), diagonal=1)
    assert (P[0, :, upper] == 0).all()
    assert (P[0, :, ~upper] >= 0).all()
    assert (P.sum(-1) - 1).abs().max().item() <= 0.01
    o_ref, _ = oracle.attention_f64(q, k, v, True)
    assert (P.double() - torch.from_numpy(o_ref)).abs().max().item() <= TOL_O_BF16


def test_query_permutation_permutes_outputs_exactly():
    a = attn()
    q, k, v = to_dev(*make_qkv(1, 2, 2, 300, 300, 128, "bf16", seed=65))
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(1)).cuda()
    o, lse = a.attn_fwd(q, k, v, causal=False)
    o2, lse2 = a.attn_fwd(q[:, :, perm].contiguous(), k, v, causal=False)
    check_status(a)
    assert torch.equal(o2, o[:, :, perm]) and torch.equal(lse2, lse[:, :, perm])


def test_kv_joint_permutation_leaves_output_unchanged():
    a = attn()
    q, k, v = to_dev(*make_qkv(1, 2, 1, 200, 300, 64, "bf16", seed=66))
    perm = torch.randperm(300, generator=torch.Generator().manual_seed(2)).cuda()
    o, lse = a.attn_fwd(q, k, v, causal=False)
    o2, lse2 = a.attn_fwd(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), causal=False)
    check_status(a)
    assert (o2.float() - o.float()).abs().max().item() <= TOL_O_BF16
    assert (lse2 - lse).abs().max().item() <= TOL_LSE_BF16


@pytest.mark.parametrize("Tq,causal", [(300, True), (1, False)])
def test_gqa_equals_repeated_mha_exactly(Tq, causal):
    a = attn()
    q, k, v = to_dev(*make_qkv(2, 8, 2, Tq, 300, 128, "bf16", seed=67))
    o, lse = (a.attn_fwd_decode(q, k, v, num_splits=2) if Tq == 1
              else a.attn_fwd(q, k, v, causal=causal))
    k4, v4 = k.repeat_interleave(4, dim=1).contiguous(), v.repeat_interleave(4, dim=1).contiguous()
    o2, lse2 = (a.attn_fwd_decode(q, k4, v4, num_splits=2) if Tq == 1
                else a.attn_fwd(q, k4, v4, causal=causal))
    check_status(a)
    if Tq == 1:  # decode: the two shapes run different head-chunk kernels
        assert (o.float() - o2.float()).abs().max().item() <= TOL_O_BF16
        assert (lse - lse2).abs().max().item() <= TOL_LSE_BF16
    else:
        assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_shift_of_keys_moves_lse_only():
    """Adding c to every K row adds scale * q_i . c to row i's scores, so the
    softmax is unchanged; the shifted keys are bf16-rounded, so the kernel is
    checked against the oracle on exactly those shifted inputs."""
    a = attn()
    q, k, v = make_qkv(1, 2, 2, 256, 256, 64, "bf16", seed=68)
    c = torch.linspace(-1, 1, 64)
    k2 = (k.float() + c).to(torch.bfloat16)
    o2, lse2 = a.attn_fwd(*to_dev(q, k2, v), causal=True)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k2, v, True)
    compare(o2, lse2, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("causal,Tq", [(True, 512), (False, 512), (False, 1)])
def test_rising_scores_take_the_exact_path(causal, Tq):
    """Scores that grow along the key axis by far more than 2^64 (in base 2)
    between the first and the last key tile force the kernels off their
    fast path (weights against the first tile's maximum) onto the exact
    max-and-rescale path; the result must still match the oracle."""
    a = attn()
    g = torch.Generator().manual_seed(69)
    Tk, D = 512, 64
    ramp = torch.linspace(0.0, 10.0, Tk)[None, None, :, None]
    q = (torch.ones(1, 2, Tq, D) + 0.3 * torch.randn(1, 2, Tq, D, generator=g)).to(torch.bfloat16)
    k = (ramp + 0.5 * torch.randn(1, 2, Tk, D, generator=g)).to(torch.bfloat16)
    v = torch.randn(1, 2, Tk, D, generator=g).to(torch.bfloat16)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, 1e-3 * max(1.0, float(abs(lse_ref).max())) / 10)


@pytest.mark.parametrize("offset", [-30.0, -12.0, 12.0, 30.0])
@pytest.mark.parametrize("causal", [True, False])
def test_first_tile_far_from_the_reference(offset, causal):
    """Every score of a row far above 2^62 or far below 2^-60 (in base 2):
    weights taken against any fixed reference such as 0 would overflow or
    vanish, so the reference must come from the row's own scores.  The
    output must still match the oracle."""
    a = attn()
    g = torch.Generator().manual_seed(70)
    T, D = 384, 64
    q = (torch.ones(1, 2, T, D) + 0.1 * torch.randn(1, 2, T, D, generator=g)).to(torch.bfloat16)
    k = (offset + 0.5 * torch.randn(1, 2, T, D, generator=g)).to(torch.bfloat16)
    v = torch.randn(1, 2, T, D, generator=g).to(torch.bfloat16)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, 1e-3 * max(1.0, float(abs(lse_ref).max())) / 10)
