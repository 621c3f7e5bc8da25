"""Problems whose tensors hold more than 2^31 elements, so that every
element offset in the kernels (O and lse rows, K/V slabs, paged block
addresses, packed rows) must be computed in 64 bits.  Parity on sampled rows
against the float64 oracle, taken one head at a time."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status

pytestmark = pytest.mark.gpu

BIG = 2 ** 31


def _randn(shape, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.bfloat16)


def _check_rows(o, lse, q, k, v, causal, picks, what):
    """picks: (b, h, i) query rows; q [B, Hq, Tq, D], k/v [B, Hkv, Tk, D]."""
    B, Hq, Tq, D = q.shape
    g = Hq // k.shape[1]
    worst_o = worst_l = 0.0
    for b, h, i in picks:
        qs = q[b:b + 1, h:h + 1].cpu()
        ks, vs = k[b:b + 1, h // g:h // g + 1].cpu(), v[b:b + 1, h // g:h // g + 1].cpu()
        o_ref, l_ref = oracle.attention_f64(qs, ks, vs, causal, rows=np.array([i]))
        worst_o = max(worst_o, float(np.abs(o[b, h, i].float().cpu().numpy() - o_ref[0]).max()))
        worst_l = max(worst_l, abs(float(lse[b, h, i]) - float(l_ref[0])))
    assert worst_o <= TOL_O_BF16, f"{what}: O error {worst_o:.3e}"
    assert worst_l <= TOL_LSE_BF16, f"{what}: lse error {worst_l:.3e}"


def test_prefill_with_q_beyond_2_31_elements():
    a = attn()
    B, Hq, Hkv, T, D = 1, 64, 8, 262144, 128   # q, o: 2^31 elements each
    assert B * Hq * T * D >= BIG
    q, k, v = _randn((B, Hq, T, D), 1), _randn((B, Hkv, T, D), 2), _randn((B, Hkv, T, D), 3)
    o, lse = a.attn_fwd(q, k, v, causal=True)
    check_status(a)
    rng = np.random.default_rng(0)
    picks = [(0, 63, T - 1), (0, 63, T - 129), (0, 40, 200000), (0, 0, 5)] + \
            [(0, int(rng.integers(Hq)), int(rng.integers(T))) for _ in range(8)]
    _check_rows(o, lse, q, k, v, True, picks, "prefill T=262144")


def test_d64_prefill_with_q_beyond_2_31_elements():
    """The head-dim-64 kernel (TMA-stored O, one query tile per item)."""
    a = attn()
    B, Hq, Hkv, T, D = 1, 128, 8, 262144, 64   # q, o: 2^31 elements each
    assert B * Hq * T * D >= BIG
    q, k, v = _randn((B, Hq, T, D), 21), _randn((B, Hkv, T, D), 22), _randn((B, Hkv, T, D), 23)
    o, lse = a.attn_fwd(q, k, v, causal=True)
    check_status(a)
    rng = np.random.default_rng(1)
    picks = [(0, 127, T - 1), (0, 127, T - 17), (0, 64, 131072), (0, 0, 3)] + \
            [(0, int(rng.integers(Hq)), int(rng.integers(T))) for _ in range(6)]
    _check_rows(o, lse, q, k, v, True, picks, "D=64 prefill T=262144")


def test_group_decode_key_ranges_with_kv_beyond_2_31_elements():
    """Eight query heads per KV head and one batch row: key ranges on the
    prefill kernel over 2^31-element K and V, merged by the combine kernel."""
    a = attn()
    B, Hq, Hkv, Tk, D = 1, 64, 8, 1 << 21, 128   # k, v: 2^31 elements each
    assert B * Hkv * Tk * D >= BIG
    q, k, v = _randn((B, Hq, 1, D), 24), _randn((B, Hkv, Tk, D), 25), _randn((B, Hkv, Tk, D), 26)
    o, lse = a.attn_fwd(q, k, v, causal=False)
    _, ranges, kernels = a.last_launch_info()
    check_status(a)
    assert ranges > 1 and kernels == 2
    _check_rows(o, lse, q, k, v, False, [(0, 63, 0), (0, 0, 0), (0, 29, 0)], "key ranges Tk=2^21")


def test_decode_with_kv_beyond_2_31_elements():
    a = attn()
    B, Hq, Hkv, Tk, D = 128, 32, 8, 16384, 128   # k, v: 2^31 elements each
    assert B * Hkv * Tk * D >= BIG
    q, k, v = _randn((B, Hq, 1, D), 4), _randn((B, Hkv, Tk, D), 5), _randn((B, Hkv, Tk, D), 6)
    o, lse = a.attn_fwd(q, k, v, causal=False)
    check_status(a)
    picks = [(127, 31, 0), (127, 0, 0), (64, 17, 0), (0, 0, 0), (100, 5, 0)]
    _check_rows(o, lse, q, k, v, False, picks, "decode Tk=16384 B=128")


def test_paged_decode_with_pool_beyond_2_31_elements():
    a = attn()
    B, Hq, Hkv, D, P, L = 128, 32, 8, 128, 16, 16384
    nblk = B * L // P + 4
    assert nblk * 2 * Hkv * P * D >= BIG
    kv = _randn((nblk, 2, Hkv, P, D), 7)
    q = _randn((B, Hq, 1, D), 8)
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(9))[: B * L // P]
    bt = perm.reshape(B, L // P).to(torch.int32).cuda()
    sl = torch.full((B,), L, dtype=torch.int32, device="cuda")
    o, lse = a.attn_fwd_decode_paged(q, kv, bt, sl)
    check_status(a)
    for b in (0, 127, 77):  # gather the request's keys on the device, then the oracle
        blk = bt[b].long()
        kb = kv[blk, 0].permute(1, 0, 2, 3).reshape(1, Hkv, L, D)
        vb = kv[blk, 1].permute(1, 0, 2, 3).reshape(1, Hkv, L, D)
        for h in (0, 31):
            o_ref, l_ref = oracle.attention_f64(q[b:b + 1, h:h + 1].cpu(),
                                                kb[:, h // 4:h // 4 + 1].cpu(),
                                                vb[:, h // 4:h // 4 + 1].cpu(), False)
            assert np.abs(o[b, h, 0].float().cpu().numpy() - o_ref[0, 0, 0]).max() <= TOL_O_BF16
            assert abs(float(lse[b, h]) - float(l_ref[0, 0, 0])) <= TOL_LSE_BF16


def test_packed_sequences_beyond_2_31_elements():
    a = attn()
    Hq, Hkv, D = 64, 8, 128
    lens = [200000, 7, 62137]
    total = sum(lens)
    assert total * Hq * D >= BIG
    q, k, v = _randn((total, Hq, D), 10), _randn((total, Hkv, D), 11), _randn((total, Hkv, D), 12)
    cu = torch.tensor([0] + lens, dtype=torch.int64).cumsum(0).to(torch.int32).cuda()
    o, lse = a.attn_fwd_varlen(q, k, v, cu, cu, True)
    check_status(a)
    starts = [0, lens[0], lens[0] + lens[1]]
    for s_idx, h, i in ((2, 63, lens[2] - 1), (2, 0, 1000), (0, 31, lens[0] - 1), (1, 5, 6)):
        r0, n = starts[s_idx], lens[s_idx]
        qs = q[r0:r0 + n, h:h + 1].permute(1, 0, 2).unsqueeze(0).cpu()
        ks = k[r0:r0 + n, h // 8:h // 8 + 1].permute(1, 0, 2).unsqueeze(0).cpu()
        vs = v[r0:r0 + n, h // 8:h // 8 + 1].permute(1, 0, 2).unsqueeze(0).cpu()
        o_ref, l_ref = oracle.attention_f64(qs, ks, vs, True, rows=np.array([i]))
        assert np.abs(o[r0 + i, h].float().cpu().numpy() - o_ref[0]).max() <= TOL_O_BF16
        assert abs(float(lse[h, r0 + i]) - float(l_ref[0])) <= TOL_LSE_BF16
