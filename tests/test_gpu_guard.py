"""Writes stay inside O and lse on every entry point: each output sits in a
buffer with sentinel-filled margins on both sides, and the margins (and, for
packed sequences, the rows no sequence covers) must be unchanged afterwards."""
import pytest
import torch

from gpu_util import attn, check_status
from transformer_attention_fwd_gb300.inputs import make_paged, make_qkv, make_varlen

pytestmark = pytest.mark.gpu

PAD = 4096


def _guarded(shape, dtype, fill):
    n = 1
    for x in shape:
        n *= x
    buf = torch.full((n + 2 * PAD,), fill, dtype=dtype, device="cuda")
    return buf, buf[PAD:PAD + n].view(*shape)


def _margins_intact(buf, fill):
    return bool((buf[:PAD] == fill).all()) and bool((buf[-PAD:] == fill).all())


@pytest.mark.parametrize("splits", [0, 5])
def test_decode_writes_stay_inside(splits):
    a = attn()
    q, k, v = (x.cuda() for x in make_qkv(3, 16, 4, 1, 2000, 128, "bf16", seed=141))
    ob, o = _guarded(q.shape, torch.bfloat16, 7.0)
    lb, lse = _guarded((3, 16, 1), torch.float32, 7.0)
    a.attn_fwd_decode(q, k, v, num_splits=splits, out=o, lse=lse)
    check_status(a)
    assert _margins_intact(ob, 7.0) and _margins_intact(lb, 7.0)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 64), (16, 8, 128)])
def test_paged_decode_writes_stay_inside(Hq, Hkv, D):
    a = attn()
    q, kv, bt, sl = (x.cuda() for x in make_paged(5, Hq, Hkv, D, 16, [300, 0, 17, 1000, 1],
                                                  seed=142))
    ob, o = _guarded(q.shape, torch.bfloat16, 7.0)
    lb, lse = _guarded((5, Hq), torch.float32, 7.0)
    a.attn_fwd_decode_paged(q, kv, bt, sl, out=o, lse=lse)
    check_status(a)
    assert _margins_intact(ob, 7.0) and _margins_intact(lb, 7.0)


def test_packed_writes_stay_inside_the_sequences():
    a = attn()
    q, k, v, cq, ck = make_varlen([130, 0, 257, 3], [200, 9, 257, 70], 8, 2, 128, seed=143)
    total = q.shape[0]
    # The offsets cover rows 0..389 of a 400-row q: rows 390..399 belong to no sequence.
    qx = torch.cat([q, torch.zeros(10, 8, 128, dtype=q.dtype)]).cuda()
    ob, o = _guarded(qx.shape, torch.bfloat16, 7.0)
    lb, lse = _guarded((8, total + 10), torch.float32, 7.0)
    a.attn_fwd_varlen(qx, k.cuda(), v.cuda(), cq.cuda(), ck.cuda(), True, out=o, lse=lse)
    check_status(a)
    assert _margins_intact(ob, 7.0) and _margins_intact(lb, 7.0)
    assert (o[total:] == 7.0).all() and (lse[:, total:] == 7.0).all()
    assert torch.isfinite(o[:total].float()).all()


def test_window_and_f16_prefill_writes_stay_inside():
    a = attn()
    for dtype, window in (("bf16", 100), ("f16", 0)):
        q, k, v = (x.cuda() for x in make_qkv(1, 4, 2, 300, 500, 64, dtype, seed=144))
        ob, o = _guarded(q.shape, q.dtype, 7.0)
        lb, lse = _guarded(q.shape[:3], torch.float32, 7.0)
        if window:
            a.attn_fwd_window(q, k, v, window, out=o, lse=lse)
        else:
            a.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
        check_status(a)
        assert _margins_intact(ob, 7.0) and _margins_intact(lb, 7.0)
