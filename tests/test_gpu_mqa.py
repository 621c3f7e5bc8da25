"""Multi-query attention (one K/V head shared by every query head, "第 11 章 ·
Attention 入门" §11.8.1 MHA / MQA / GQA) on the prefill, decode and packed
paths, against the float64 oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import (TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, to_dev)
from transformer_attention_fwd_gb300.inputs import make_qkv, make_varlen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_mqa_prefill(D, causal):
    a = attn()
    q, k, v = make_qkv(2, 16, 1, 300, 300, D, "bf16", seed=91)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"MQA prefill D{D}")


@pytest.mark.parametrize("Hq", [8, 32, 64])
@pytest.mark.parametrize("splits", [0, 3])
def test_mqa_decode(Hq, splits):
    a = attn()
    q, k, v = make_qkv(4, Hq, 1, 1, 1000, 128, "bf16", seed=92)
    o, lse = a.attn_fwd_decode(*to_dev(q, k, v), num_splits=splits)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"MQA decode Hq{Hq} splits{splits}")


def test_mqa_varlen():
    a = attn()
    q, k, v, cq, ck = make_varlen([200, 7, 129], [200, 50, 300], 12, 1, 128, seed=93)
    o, lse = a.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), True)
    check_status(a)
    o_ref, lse_ref = oracle.attention_varlen_f64(q, k, v, cq, ck, True)
    assert np.abs(o.float().cpu().numpy() - o_ref).max() <= TOL_O_BF16
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= TOL_LSE_BF16
