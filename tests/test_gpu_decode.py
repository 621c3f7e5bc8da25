"""Split-KV decode parity against the float64 oracle."""
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gqa_decode_full(seed):
    """B=64, Hq=32, Hkv=8, Tk=4096, D=128: every output compared."""
    a = attn()
    w = WORKLOADS["gqa_decode_bf16_b64_hq32_hkv8_tk4096_d128"]
    q, k, v = make_workload(w, seed)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=False)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, w.name)


def test_split_count_does_not_change_result():
    a = attn()
    q, k, v = to_dev(*make_qkv(4, 8, 2, 1, 3000, 128, "bf16", seed=3))
    ref_o, ref_l = a.attn_fwd_decode(q, k, v, num_splits=1)
    for s in (2, 3, 4, 8, 16, 64):
        o, l = a.attn_fwd_decode(q, k, v, num_splits=s)
        assert (o.float() - ref_o.float()).abs().max().item() <= 8e-3, s
        assert (l - ref_l).abs().max().item() <= 2e-5, s
    check_status(a)


def test_decode_equals_prefill_kernel_at_tq1():
    a = attn()
    q, k, v = to_dev(*make_qkv(2, 8, 4, 1, 777, 128, "bf16", seed=4))
    o1, l1 = a.attn_fwd_decode(q, k, v)
    o2, l2 = a.attn_fwd_prefill(q, k, v, causal=True)
    check_status(a)
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 5e-5


@pytest.mark.parametrize("B,Hq,Hkv,Tk,D,splits", [
    (1, 1, 1, 1, 64, 0), (3, 4, 4, 7, 64, 0), (2, 32, 1, 1000, 128, 0),  # MHA tiny, MQA
    (2, 16, 2, 4097, 128, 0), (1, 8, 8, 513, 64, 5), (2, 12, 4, 129, 128, 1),
    (1, 6, 2, 2000, 64, 7),
    (2, 64, 8, 1500, 64, 0), (3, 64, 8, 777, 128, 0),  # eight heads per KV head: two warp groups
])
def test_decode_shapes(B, Hq, Hkv, Tk, D, splits):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, 1, Tk, D, "bf16", seed=Tk)
    o, lse = a.attn_fwd_decode(*to_dev(q, k, v), num_splits=splits)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gqa8_decode_full(seed):
    """B=32, Hq=64, Hkv=8, Tk=4096, D=128 (eight query heads per KV head):
    automatic mode runs the tensor-core prefill kernel on the query-head
    groups (one work item per (b, hkv)); every output compared."""
    a = attn()
    w = WORKLOADS["gqa8_decode_bf16_b32_hq64_hkv8_tk4096_d128"]
    q, k, v = make_workload(w, seed)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=False)
    _, items, kernels = a.last_launch_info()
    check_status(a)
    assert items == w.B * w.Hkv and kernels == 1
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, w.name)


def _group_route(B, Hq, Hkv, Tk, D, dtype, sms):
    """The automatic decode route for 8 or more query heads per KV head, as
    the library states it: key ranges on the prefill kernel (D=128,
    (b, hkv) pairs filling at most half the SMs, two key tiles per range),
    else the prefill kernel per (b, hkv) from B*Hq >= 512 rows on, else the
    CUDA-core stream-K kernel."""
    pairs, tiles = B * Hkv, -(-Tk // 128)
    if D == 128 and 2 * pairs <= sms:
        splits = min(sms // pairs, tiles // 2)
        if splits >= 2:
            per = -(-tiles // splits)
            return "split", -(-tiles // per)
    if B * Hq >= 512:
        return "prefill", B * Hkv * -(-(Hq // Hkv) // (128 if D == 64 else 256))
    return "stream", 0


@pytest.mark.parametrize("B,Hq,Hkv,Tk,D,dtype", [
    (8, 64, 8, 1000, 128, "bf16"),    # 64 pairs: two key ranges each
    (4, 64, 8, 4096, 128, "bf16"),    # 32 pairs: four key ranges each
    (2, 64, 8, 32768, 128, "bf16"),   # long keys, nine ranges
    (1, 32, 1, 8192, 128, "bf16"),    # MQA, one pair: 32 ranges
    (16, 32, 2, 513, 128, "bf16"),    # sixteen heads per KV head, a ragged last tile
    (1, 512, 1, 2048, 128, "bf16"),   # 512 query heads: two query blocks per range
    (16, 64, 8, 700, 128, "bf16"),    # 128 pairs: one item per (b, hkv)
    (4, 128, 8, 3001, 64, "bf16"),    # D=64 (two CTAs per SM), one item per (b, hkv)
    (16, 64, 8, 700, 128, "f16"),     # fp16: one item per (b, hkv)
    (2, 64, 8, 1000, 128, "f16"),     # fp16 with few rows: key ranges
    (2, 64, 8, 1000, 64, "bf16"),     # D=64 with few rows: the CUDA-core kernel
])
def test_many_heads_per_kv_head_decode(B, Hq, Hkv, Tk, D, dtype):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, 1, Tk, D, dtype, seed=Tk + Hq)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=False)
    _, items, kernels = a.last_launch_info()
    check_status(a)
    route, n = _group_route(B, Hq, Hkv, Tk, D, dtype,
                            torch.cuda.get_device_properties(0).multi_processor_count)
    if route == "split":
        assert (items, kernels) == (n, 2)
    elif route == "prefill":
        assert (items, kernels) == (n, 1)
    else:
        assert items == 0
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"{route} route")


def test_prefill_route_agrees_with_split_kernel():
    """The two decode kernels for eight heads per KV head agree (an explicit
    split count keeps the CUDA-core split kernel)."""
    a = attn()
    q, k, v = to_dev(*make_qkv(8, 64, 8, 1, 2500, 128, "bf16", seed=9))
    o1, l1 = a.attn_fwd_decode(q, k, v)
    o2, l2 = a.attn_fwd_decode(q, k, v, num_splits=4)
    check_status(a)
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 5e-5
