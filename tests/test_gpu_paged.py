"""Decode over a paged KV cache against the float64 oracle ("第 11 章 ·
Attention 入门", 11.11, the KV-cache / VMM passage)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import (PAGED_WORKLOADS, make_paged,
                                                    make_paged_workload)

pytestmark = pytest.mark.gpu


def _run(a, q, kv, bt, sl):
    o, lse = a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    check_status(a)
    return o[:, :, 0, :], lse


def _check(a, q, kv, bt, sl, what):
    o, lse = _run(a, q, kv, bt, sl)
    o_ref, lse_ref = oracle.decode_paged_f64(q, kv, bt, sl)
    empty = (sl == 0).numpy()
    if empty.any():  # requests without keys: O = 0, lse = -inf exactly
        assert (o[torch.from_numpy(empty).cuda()] == 0).all()
        assert torch.isneginf(lse[torch.from_numpy(empty).cuda()]).all()
        keep = ~empty
        o, lse = o[torch.from_numpy(keep).cuda()], lse[torch.from_numpy(keep).cuda()]
        o_ref, lse_ref = o_ref[keep], lse_ref[keep]
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, what)


@pytest.mark.parametrize("B,Hq,Hkv,D,page,lens", [
    (3, 8, 2, 128, 16, [1, 17, 300]),
    (4, 16, 16, 64, 8, [5, 64, 0, 129]),          # MHA, D=64, an empty request
    (2, 8, 1, 128, 32, [1000, 33]),               # MQA
    (5, 32, 8, 128, 16, [4096, 1, 2048, 15, 16]),
    (3, 4, 2, 64, 1, [3, 40, 7]),                 # one token per block
    (2, 8, 2, 128, 256, [700, 256]),              # large blocks
    (2, 16, 2, 64, 16, [100, 2000]),              # eight heads per KV head, D=64
    (2, 8, 4, 128, 32, [700, 33]),                # 32-token blocks, lengths off the block size
    (3, 16, 8, 128, 8, [1000, 9, 64]),            # 8-token blocks: eight pages per 64-key chunk
    (2, 8, 8, 128, 16, [300, 4096]),              # MHA in 16-token blocks
    (2, 32, 8, 64, 16, [777, 2048]),              # D=64, GQA-4
    (2, 8, 4, 64, 32, [500, 31]),                 # D=64, 32-token blocks
    (3, 8, 2, 128, 16, [0, 0, 0]),                # no request has keys
    (4, 8, 2, 128, 16, [0, 300, 0, 5]),           # empty requests around short ones
])
def test_paged_matches_oracle(B, Hq, Hkv, D, page, lens):
    a = attn()
    q, kv, bt, sl = make_paged(B, Hq, Hkv, D, page, lens, seed=11)
    _check(a, q, kv, bt, sl, f"B{B} Hq{Hq} Hkv{Hkv} D{D} P{page} {lens}")


def test_many_short_requests():
    """Hundreds of units per SM slice: most units are finished inside one CTA."""
    a = attn()
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 200, size=96)
    q, kv, bt, sl = make_paged(96, 4, 4, 64, 16, lens, seed=12)
    _check(a, q, kv, bt, sl, "96 short requests")


def test_many_short_requests_gqa():
    """Short GQA requests in 16-token pages: slices start and end inside pages
    and units of several requests share a CTA."""
    a = attn()
    rng = np.random.default_rng(17)
    lens = rng.integers(1, 200, size=80)
    q, kv, bt, sl = make_paged(80, 16, 8, 128, 16, lens, seed=17)
    _check(a, q, kv, bt, sl, "80 short GQA requests")


@pytest.mark.parametrize("B,D,dtype", [(1024, 64, "bf16"), (1025, 64, "bf16"), (1500, 64, "bf16"),
                                       (1100, 128, "f16")])
def test_length_prefix_in_the_kernel_and_in_a_prefix_kernel(B, D, dtype):
    """Up to 1024 requests every CTA sums the lengths itself (two kernels: the
    stream kernel and the combine); more take a prefix kernel first."""
    a = attn()
    rng = np.random.default_rng(B)
    lens = rng.integers(0, 120, size=B)
    lens[::97] = 0
    q, kv, bt, sl = make_paged(B, 4, 2, D, 16, lens, seed=B, dtype=dtype)
    _check(a, q, kv, bt, sl, f"{B} requests")
    _, _, kernels = a.last_launch_info()
    assert kernels == (2 if B <= 1024 else 3)
    sl[B // 2] = -1  # a bad length is reported on both paths
    a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT


@pytest.mark.parametrize("seed", [0, 1])
def test_paged_bench_workload_full(seed):
    """B=64, Hq=32, Hkv=8, 4096 keys each in 16-token blocks: every output."""
    a = attn()
    w = PAGED_WORKLOADS["gqa_paged_decode_bf16_b64_hq32_hkv8_tk4096_d128_p16"]
    q, kv, bt, sl = make_paged_workload(w, seed)
    _check(a, q, kv, bt, sl, w.name)


def test_contiguous_blocks_equal_dense_decode():
    """Blocks in token order hold the dense cache; the paged call then agrees
    with the dense decode call on the dense tensors."""
    a = attn()
    B, Hq, Hkv, D, P, L = 4, 16, 4, 128, 16, 1000
    g = torch.Generator().manual_seed(13)
    q = torch.randn(B, Hq, 1, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, L, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, L, D, generator=g).to(torch.bfloat16)
    npg = -(-L // P)
    kv = torch.zeros(B * npg, 2, Hkv, P, D, dtype=torch.bfloat16)
    for b in range(B):
        for pg in range(npg):
            t0, t1 = pg * P, min(L, pg * P + P)
            kv[b * npg + pg, 0, :, : t1 - t0] = k[b, :, t0:t1]
            kv[b * npg + pg, 1, :, : t1 - t0] = v[b, :, t0:t1]
    bt = torch.arange(B * npg, dtype=torch.int32).reshape(B, npg)
    sl = torch.full((B,), L, dtype=torch.int32)
    o, lse = _run(a, q, kv, bt, sl)
    od, ld = a.attn_fwd_decode(*to_dev(q, k, v))
    check_status(a)
    assert (o.float() - od[:, :, 0].float()).abs().max().item() <= 8e-3
    assert (lse - ld[:, :, 0]).abs().max().item() <= 2e-5


def test_rows_past_the_end_and_spare_blocks_are_never_read():
    a = attn()
    lens = [5, 33, 16]
    q, kv, bt, sl = make_paged(3, 8, 2, 128, 16, lens, seed=14, spare_blocks=4)
    used = set()
    for b, L in enumerate(lens):
        for t in range(L):
            used.add((int(bt[b, t // 16]), t % 16))
    poison = torch.full_like(kv[0, 0, 0, 0], float("nan"))
    for blk in range(kv.shape[0]):
        for r in range(16):
            if (blk, r) not in used:
                kv[blk, :, :, r] = poison
    _check(a, q, kv, bt, sl, "poisoned unused rows")


def test_bad_block_id_is_reported_and_context_stays_usable():
    a = attn()
    q, kv, bt, sl = make_paged(2, 8, 2, 128, 16, [40, 20], seed=15)
    bt[1, 0] = kv.shape[0] + 7  # outside the pool
    a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    bt[1, 0] = -2
    a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    q, kv, bt, sl = make_paged(2, 8, 2, 128, 16, [40, 20], seed=15)
    _check(a, q, kv, bt, sl, "after a reported bad block id")


def test_bad_length_is_reported():
    a = attn()
    q, kv, bt, sl = make_paged(2, 8, 2, 128, 16, [40, 20], seed=16)
    sl[0] = bt.shape[1] * 16 + 1  # longer than the table
    a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
    sl[0] = -3
    a.attn_fwd_decode_paged(*to_dev(q, kv, bt, sl))
    assert a.device_status() == a.ATTN_ERR_BAD_INPUT
