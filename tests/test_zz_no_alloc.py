"""attn_fwd_decode_noalloc: the decode entry point that allocates nothing.

It exists for callers that cannot let a library allocate device memory in the
middle of a call (engines that reserve all of HBM for their own allocator, or
that keep allocation out of a latency-critical decode step).  Its partial
results live in a fixed 8 MiB workspace inside the library instead of memory
allocated per call.  Here it is called straight through the C ABI, twice in a
row with different shapes, and each result is checked against the allocating
entry point attn_fwd_decode within the parity tolerances the other decode
tests use.  This file sorts last so that a run stopping at its first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


def _noalloc():
    a = attn()
    fn = ctypes.CDLL(a.LIB_PATH).attn_fwd_decode_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, P]
    fn.restype = ctypes.c_int
    return a, fn


def _call(fn, q, k, v, splits):
    B, Hq, _, D = q.shape
    _, Hkv, Tk, _ = k.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device="cuda")
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
            Tk, D, D ** -0.5, splits, torch.cuda.current_stream().cuda_stream)
    return st, o, lse


def test_noalloc_decode_matches_allocating_decode_on_two_calls():
    a, fn = _noalloc()
    cases = [(16, 32, 8, 4096, 128, 0), (4, 12, 4, 3001, 64, 5)]
    outs = []
    for i, (B, Hq, Hkv, Tk, D, splits) in enumerate(cases):
        q, k, v = to_dev(*make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=20 + i))
        st, o, lse = _call(fn, q, k, v, splits)
        assert st == a.ATTN_OK, a.last_error()
        outs.append((q, k, v, splits, o, lse))
    torch.cuda.synchronize()
    check_status(a)
    for q, k, v, splits, o, lse in outs:
        o_ref, lse_ref = a.attn_fwd_decode(q, k, v, num_splits=splits)
        check_status(a)
        assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O_BF16
        assert (lse - lse_ref).abs().max().item() <= TOL_LSE_BF16


def test_noalloc_rejects_partials_beyond_the_static_workspace():
    a, fn = _noalloc()
    B, Hq, Hkv, Tk, D = 64, 32, 8, 4096, 128
    q, k, v = to_dev(*make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=30))
    splits = 16  # 64*32*16*129*4 bytes > 8 MiB
    assert B * Hq * splits * (D + 1) * 4 > SCRATCH_BYTES
    st, _, _ = _call(fn, q, k, v, splits)
    assert st == a.ATTN_ERR_UNSUPPORTED
    assert "static workspace" in a.last_error()
    st, o, lse = _call(fn, q, k, v, 0)  # automatic mode: the stream-K fragments fit
    assert st == a.ATTN_OK, a.last_error()
    o_ref, lse_ref = a.attn_fwd_decode(q, k, v)
    check_status(a)
    assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O_BF16
    assert (lse - lse_ref).abs().max().item() <= TOL_LSE_BF16


def _stream_fits(B, Hq, Hkv, Tk, D, num_sms):
    """Whether the stream-K fragments fit in the static workspace (the sizing
    the header states for automatic mode)."""
    group = Hq // Hkv
    hc = next(h for h in (8, 4, 2, 1) if group % h == 0)
    total = B * Hkv * (group // hc) * Tk
    per = -(-total // num_sms)
    nseg = -(-Tk // per) + 1
    return B * Hq * nseg * (D + 1) * 4 + 256 <= SCRATCH_BYTES


@pytest.mark.parametrize("B,expect_stream", [(254, True), (255, False)])
def test_noalloc_automatic_mode_uses_stream_k_while_it_fits(B, expect_stream):
    a, fn = _noalloc()
    Hq, Hkv, Tk, D = 32, 8, 256, 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _stream_fits(B, Hq, Hkv, Tk, D, sms) == expect_stream
    q, k, v = to_dev(*make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=40 + B))
    st, o, lse = _call(fn, q, k, v, 0)
    assert st == a.ATTN_OK, a.last_error()
    grid, items, _ = a.last_launch_info()
    torch.cuda.synchronize()
    check_status(a)
    o_ref, lse_ref = a.attn_fwd_decode(q, k, v)
    grid_ref, _, _ = a.last_launch_info()
    check_status(a)
    if expect_stream:
        # The same kernels on the same slices as attn_fwd_decode: equal bits.
        assert grid == grid_ref <= sms and items == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    else:
        # The split kernel: one CTA row per (b, hkv), tolerance of the split path.
        assert grid == B * Hkv and items >= 1
        assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O_BF16
        assert (lse - lse_ref).abs().max().item() <= TOL_LSE_BF16


@pytest.mark.parametrize("B,Hq,Hkv,Tk,D,splits", [
    (16, 32, 8, 4096, 128, 0),   # automatic mode: stream-K, fragments in the array
    (4, 12, 4, 3001, 64, 5),     # explicit count: the split kernel, partials in the array
])
def test_noalloc_decode_matches_the_oracle(B, Hq, Hkv, Tk, D, splits):
    """Each of the two kernels this entry point runs, compared directly with
    the float64 oracle on the same bf16 inputs."""
    a, fn = _noalloc()
    qc, kc, vc = make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=50 + D)
    q, k, v = to_dev(qc, kc, vc)
    st, o, lse = _call(fn, q, k, v, splits)
    assert st == a.ATTN_OK, a.last_error()
    _, items, _ = a.last_launch_info()
    check_status(a)
    assert (items == 0) == (splits == 0)  # stream-K reports no split count
    o_ref, lse_ref = oracle.attention_f64(qc, kc, vc, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"noalloc splits={splits}")


def _randn_dev(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.bfloat16)


@pytest.mark.parametrize("B,Tk,lowered", [
    (32, 8192, False),   # automatic count (4 splits) fits the array as chosen
    (128, 1024, True),   # automatic count needs more than 8 MiB: lowered until it fits
])
def test_noalloc_automatic_mode_for_mha_uses_the_array(B, Tk, lowered):
    """MHA (Hq == Hkv) in automatic mode runs the split kernel with more than
    one split, so its partials live in the static array; where the count
    attn_fwd_decode would choose does not fit, the count is lowered."""
    a, fn = _noalloc()
    Hq = Hkv = 32
    D = 128
    q = _randn_dev((B, Hq, 1, D), 60 + B)
    k = _randn_dev((B, Hkv, Tk, D), 61 + B)
    v = _randn_dev((B, Hkv, Tk, D), 62 + B)
    o_ref, lse_ref = a.attn_fwd_decode(q, k, v)
    _, splits_ref, _ = a.last_launch_info()
    check_status(a)
    ref_bytes = B * Hq * splits_ref * (D + 1) * 4
    assert splits_ref > 1
    assert (ref_bytes > SCRATCH_BYTES) == lowered, (splits_ref, ref_bytes)
    for call in range(2):  # twice: the array keeps the first call's partials
        st, o, lse = _call(fn, q, k, v, 0)
        assert st == a.ATTN_OK, a.last_error()
        _, splits, _ = a.last_launch_info()
        check_status(a)
        assert 1 < splits <= splits_ref
        assert B * Hq * splits * (D + 1) * 4 <= SCRATCH_BYTES
        if lowered:
            assert splits < splits_ref
            assert (o.float() - o_ref.float()).abs().max().item() <= TOL_O_BF16
            assert (lse - lse_ref).abs().max().item() <= TOL_LSE_BF16
        else:  # the same kernels with the same split count: equal bits
            assert splits == splits_ref
            assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("B,Hq,Hkv,Tk", [
    (4, 64, 8, 4096),    # few (b, hkv) pairs: key ranges on the prefill kernel, partials in the array
    (32, 64, 8, 1000),   # enough pairs: the prefill kernel per (b, hkv), no workspace at all
])
def test_noalloc_wide_groups_match_the_allocating_decode(B, Hq, Hkv, Tk):
    """Eight query heads per KV head: automatic mode runs the same tensor-core
    kernels as attn_fwd_decode (equal bits), twice in a row."""
    a, fn = _noalloc()
    D = 128
    qc, kc, vc = make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=70 + B)
    q, k, v = to_dev(qc, kc, vc)
    o_ref, lse_ref = a.attn_fwd_decode(q, k, v)
    info_ref = a.last_launch_info()
    check_status(a)
    for call in range(2):
        st, o, lse = _call(fn, q, k, v, 0)
        assert st == a.ATTN_OK, a.last_error()
        assert a.last_launch_info() == info_ref
        check_status(a)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    o64, lse64 = oracle.attention_f64(qc, kc, vc, False)
    compare(o, lse, o64, lse64, TOL_O_BF16, TOL_LSE_BF16, "noalloc, eight heads per KV head")
