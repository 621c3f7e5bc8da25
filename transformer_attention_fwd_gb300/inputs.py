"""Seeded synthetic inputs and the named workloads.

This module is shared by the tests, the bench and the smoke check.  It holds
no attention arithmetic: it only draws Q, K, V from N(0, 1) with a seeded CPU
generator and, for bf16 workloads, rounds them to bf16 (round-to-nearest-even,
torch's ``.to(torch.bfloat16)``).  Both the CUDA library and the oracle are fed
exactly these values.

Layouts are [B, H, T, D] row-major with D innermost; query tensors carry Hq
heads and key/value tensors Hkv heads ("3.3 Self-Attention机制深入理解" §4.2,
the (batch, num_heads, seq_len, head_dim) layout after the transpose).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tk: int
    D: int
    causal: bool
    dtype: str  # "f32" or "bf16"

    @property
    def flops(self) -> float:
        """4*B*Hq*Tq*Tk*D, halved when causal (the metric's convention)."""
        f = 4.0 * self.B * self.Hq * self.Tq * self.Tk * self.D
        return f / 2.0 if self.causal else f

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once, lse (fp32)."""
        e = self.elem_bytes
        q = self.B * self.Hq * self.Tq * self.D * e
        kv = 2 * self.B * self.Hkv * self.Tk * self.D * e
        o = q
        lse = self.B * self.Hq * self.Tq * 4
        return q + kv + o + lse


# The five named workloads (plus the non-causal variants the tests also run).
WORKLOADS = {
    "sdpa_f32_b1_h1_t128_d64_causal":
        Workload("sdpa_f32_b1_h1_t128_d64_causal", 1, 1, 1, 128, 128, 64, True, "f32"),
    "sdpa_f32_b1_h4_t128_d64_causal":
        Workload("sdpa_f32_b1_h4_t128_d64_causal", 1, 4, 4, 128, 128, 64, True, "f32"),
    "sdpa_f32_b1_h4_t128_d64_noncausal":
        Workload("sdpa_f32_b1_h4_t128_d64_noncausal", 1, 4, 4, 128, 128, 64, False, "f32"),
    "gpt2s_prefill_bf16_b8_h12_t1024_d64_causal":
        Workload("gpt2s_prefill_bf16_b8_h12_t1024_d64_causal", 8, 12, 12, 1024, 1024, 64, True, "bf16"),
    "llama3_8b_prefill_bf16_b1_hq32_hkv8_t8192_d128_causal":
        Workload("llama3_8b_prefill_bf16_b1_hq32_hkv8_t8192_d128_causal", 1, 32, 8, 8192, 8192, 128, True, "bf16"),
    "llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_noncausal":
        Workload("llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_noncausal", 1, 32, 8, 4096, 4096, 128, False, "bf16"),
    # Half-length causal variant, used for small ncu captures of the prefill kernel.
    "llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_causal":
        Workload("llama3_8b_prefill_bf16_b1_hq32_hkv8_t4096_d128_causal", 1, 32, 8, 4096, 4096, 128, True, "bf16"),
    "gqa_decode_bf16_b64_hq32_hkv8_tk4096_d128":
        Workload("gqa_decode_bf16_b64_hq32_hkv8_tk4096_d128", 64, 32, 8, 1, 4096, 128, False, "bf16"),
}


def torch_dtype(dtype: str) -> torch.dtype:
    if dtype == "f32":
        return torch.float32
    if dtype == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown dtype {dtype!r}")


def make_qkv(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, D: int,
             dtype: str = "bf16", seed: int = 0):
    """Draw Q [B,Hq,Tq,D], K and V [B,Hkv,Tk,D] iid N(0,1) on the CPU.

    One ``torch.Generator`` seeded with ``seed`` draws Q, then K, then V in
    float32; bf16 workloads then round each tensor to bf16 (RNE).  Returns CPU
    tensors in the I/O dtype.
    """
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn(B, Hq, Tq, D, generator=g, dtype=torch.float32)
    k = torch.randn(B, Hkv, Tk, D, generator=g, dtype=torch.float32)
    v = torch.randn(B, Hkv, Tk, D, generator=g, dtype=torch.float32)
    td = torch_dtype(dtype)
    if td != torch.float32:
        q, k, v = q.to(td), k.to(td), v.to(td)
    return q, k, v


def make_workload(w: Workload, seed: int = 0):
    return make_qkv(w.B, w.Hq, w.Hkv, w.Tq, w.Tk, w.D, w.dtype, seed)
