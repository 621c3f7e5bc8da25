"""bf16 tensor-core prefill parity against the float64 oracle run on the same
bf16-rounded inputs (max abs error 1e-2 on O, 1e-4 on lse)."""
import pytest
import torch

import oracle
from gpu_util import TOL_LSE_BF16, TOL_O_BF16, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,D,causal", [
    (1, 1, 1, 128, 128, 64, False),     # one tile
    (1, 1, 1, 128, 128, 128, True),
    (1, 2, 1, 256, 256, 64, True),      # one full work item, GQA
    (1, 2, 2, 300, 300, 128, True),     # ragged tail, several tiles
    (2, 4, 2, 300, 300, 64, False),
    (1, 4, 1, 513, 513, 128, True),     # MQA, ragged
    (1, 2, 1, 200, 520, 128, True),     # Tq < Tk, bottom-right causal
    (1, 3, 3, 1, 77, 64, True),         # Tq = 1 through the prefill kernel
    (1, 2, 2, 5, 5, 64, True),          # tiny
    (2, 2, 1, 700, 130, 64, False),     # Tk barely past one tile
])
def test_prefill_small_shapes(B, Hq, Hkv, Tq, Tk, D, causal):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, D, "bf16", seed=Tq * 7 + Tk)
    o, lse = a.attn_fwd_prefill(*to_dev(q, k, v), causal=causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,dtype", [
    (1, 32, 8, 1024, 1024, "bf16"),   # 128 work items of 8 key tiles (fewer than the SMs)
    (1, 8, 2, 256, 8192, "bf16"),     # 8 items of 64 key tiles
    (1, 40, 4, 777, 1500, "bf16"),    # ragged query and key tails, 160 items
    (2, 5, 1, 100, 3000, "f16"),      # fewer rows than an item, MQA, fp16
    (1, 19, 19, 512, 640, "bf16"),    # 38 items of 5 key tiles
    (1, 1, 1, 128, 512, "bf16"),      # one item
    (1, 38, 2, 1024, 1024, "bf16"),   # 152 items: one whole wave
])
def test_noncausal_shapes(B, Hq, Hkv, Tq, Tk, dtype):
    """Non-causal prefill at D=128 over item counts below, at and above one
    wave of SMs, with ragged tails: one kernel, every output compared."""
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, 128, dtype, seed=Tq + Tk)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=False)
    _, _, kernels = a.last_launch_info()
    check_status(a)
    assert kernels == 1
    o_ref, lse_ref = oracle.attention_f64(q, k, v, False)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"non-causal {B} {Hq} {Tq} {Tk}")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gpt2_small_prefill_full(seed):
    """B=8, H=12, T=1024, D=64 causal: every output compared."""
    a = attn()
    w = WORKLOADS["gpt2s_prefill_bf16_b8_h12_t1024_d64_causal"]
    q, k, v = make_workload(w, seed)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=True)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, True)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, w.name)


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", ["llama3_8b_prefill_bf16_b1_hq32_hkv8_t8192_d128_causal",
                                  "llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_noncausal"])
def test_llama3_prefill_full(name, seed):
    """Full-size GQA prefill (Hq=32, Hkv=8, D=128; T=8192 causal and T=4096
    non-causal): every output row compared with the float64 oracle, which
    takes a few seconds per seed on the host's cores."""
    a = attn()
    w = WORKLOADS[name]
    q, k, v = make_workload(w, seed)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=w.causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, w.causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16, f"{name} seed {seed}")


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,D,causal", [
    (1, 4, 4, 4096, 4096, 64, False),   # 32 key tiles per work item
    (2, 8, 2, 2048, 2048, 64, True),    # GQA, many items per CTA
    (3, 6, 3, 1000, 1777, 64, True),    # Tq < Tk: limits cross 32-key chunks
])
def test_d64_longer_sequences(B, Hq, Hkv, Tq, Tk, D, causal):
    """Head dim 64 runs two CTAs per SM on one query tile each; longer key
    walks and several items per CTA cycle every pipeline barrier."""
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, D, "bf16", seed=Tq + Tk)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_BF16, TOL_LSE_BF16)


@pytest.mark.parametrize("T,D", [(300, 128), (300, 64), (1, 64), (33, 64)])
def test_prefill_output_guard_bands(T, D):
    """Writes stay inside O and lse: sentinel margins around both are untouched
    (the head-dim-64 kernel writes O with TMA stores of 32-row boxes, which
    must leave out the rows past Tq)."""
    a = attn()
    B, Hq, Hkv = 1, 2, 1
    q, k, v = to_dev(*make_qkv(B, Hq, Hkv, T, T, D, "bf16", seed=5))
    n, pad = B * Hq * T * D, 4096
    o_buf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * Hq * T + 2 * pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + n].view(B, Hq, T, D)
    lse = l_buf[pad:pad + B * Hq * T].view(B, Hq, T)
    a.attn_fwd_prefill(q, k, v, causal=True, out=o, lse=lse)
    check_status(a)
    assert (o_buf[:pad] == 7.0).all() and (o_buf[pad + n:] == 7.0).all()
    assert (l_buf[:pad] == 7.0).all() and (l_buf[pad + B * Hq * T:] == 7.0).all()
