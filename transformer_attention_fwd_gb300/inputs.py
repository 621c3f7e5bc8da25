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
    # Eight query heads per KV head (a larger query-head group than the named
    # decode workload's four; "3.3 Self-Attention机制深入理解" §9.3's group map).
    "gqa8_decode_bf16_b32_hq64_hkv8_tk4096_d128":
        Workload("gqa8_decode_bf16_b32_hq64_hkv8_tk4096_d128", 32, 64, 8, 1, 4096, 128, False, "bf16"),
}


def torch_dtype(dtype: str) -> torch.dtype:
    if dtype == "f32":
        return torch.float32
    if dtype == "bf16":
        return torch.bfloat16
    if dtype == "f16":
        return torch.float16
    raise ValueError(f"unknown dtype {dtype!r}")


def make_qkv(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, D: int,
             dtype: str = "bf16", seed: int = 0):
    """Draw Q [B,Hq,Tq,D], K and V [B,Hkv,Tk,D] iid N(0,1) on the CPU.

    One ``torch.Generator`` seeded with ``seed`` draws Q, then K, then V in
    float32; bf16 (fp16) workloads then round each tensor to bf16 (fp16), RNE.
    Returns CPU tensors in the I/O dtype.
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


@dataclass(frozen=True)
class PagedWorkload:
    """Decode against a paged KV cache: B requests of `seq_len` keys each in
    blocks of `page` tokens ("第 11 章 · Attention 入门", 11.11, the KV-cache /
    VMM passage: 16-token blocks holding K and V for all KV heads)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    seq_len: int
    D: int
    page: int

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: every cached K/V row of the requests once, Q,
        O (bf16) and lse (fp32); the block table and lengths are not counted."""
        q = self.B * self.Hq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.seq_len * self.D * 2
        return q + kv + q + self.B * self.Hq * 4


PAGED_WORKLOADS = {
    "gqa_paged_decode_bf16_b64_hq32_hkv8_tk4096_d128_p16":
        PagedWorkload("gqa_paged_decode_bf16_b64_hq32_hkv8_tk4096_d128_p16", 64, 32, 8, 4096, 128, 16),
}


def make_paged(B: int, Hq: int, Hkv: int, D: int, page: int, seq_lens, seed: int = 0,
               spare_blocks: int = 3, max_pages: int | None = None, dtype: str = "bf16"):
    """Draw a paged-cache decode problem on the CPU.

    q [B, Hq, 1, D] and the block pool kv [num_blocks, 2, Hkv, page, D] are iid
    N(0, 1) rounded to bf16 (or fp16 with dtype="f16"); the pool has the blocks the requests need plus
    `spare_blocks` unreferenced ones.  Request b's pages get distinct blocks in
    a seeded random order; block-table entries past a request's last page are
    -1 (never valid).  Returns (q, kv, block_table int32 [B, max_pages],
    seq_lens int32 [B]).
    """
    g = torch.Generator().manual_seed(int(seed))
    lens = [int(x) for x in seq_lens]
    pages = [-(-L // page) for L in lens]
    if max_pages is None:
        max_pages = max(1, max(pages))
    nblk = sum(pages) + spare_blocks
    td = torch_dtype(dtype)
    q = torch.randn(B, Hq, 1, D, generator=g, dtype=torch.float32).to(td)
    kv = torch.randn(nblk, 2, Hkv, page, D, generator=g, dtype=torch.float32).to(td)
    perm = torch.randperm(nblk, generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        table[b, :pages[b]] = perm[nxt:nxt + pages[b]].to(torch.int32)
        nxt += pages[b]
    return q, kv, table, torch.tensor(lens, dtype=torch.int32)


def make_paged_workload(w: PagedWorkload, seed: int = 0):
    return make_paged(w.B, w.Hq, w.Hkv, w.D, w.page, [w.seq_len] * w.B, seed)


@dataclass(frozen=True)
class VarlenWorkload:
    """Prefill of `n_seq` sequences of mixed length packed along the token
    axis ((T, H, D) tensors, "第 11 章 · Attention 入门", 11.11).  Lengths are
    drawn log-uniformly in [min_len, max_len] from a seeded generator, so short
    and long sequences share one launch; each sequence attends only to itself
    (Tq = Tk per sequence)."""
    name: str
    n_seq: int
    min_len: int
    max_len: int
    Hq: int
    Hkv: int
    D: int
    causal: bool
    len_seed: int = 0

    def seqlens(self) -> list[int]:
        g = torch.Generator().manual_seed(int(self.len_seed))
        u = torch.rand(self.n_seq, generator=g, dtype=torch.float64)
        lo, hi = torch.log(torch.tensor(float(self.min_len))), torch.log(torch.tensor(float(self.max_len)))
        return [int(x) for x in torch.exp(lo + u * (hi - lo)).round().to(torch.int64)]

    def flops(self) -> float:
        """Score and P.V multiply-adds, 4 flops per visible (query, key) pair
        and head dimension, with the causal pair count taken as T^2 / 2."""
        pairs = sum(L * L * (0.5 if self.causal else 1.0) for L in self.seqlens())
        return 4.0 * pairs * self.D * self.Hq


VARLEN_WORKLOADS = {
    "llama3_8b_varlen_prefill_bf16_32seq_len128to8192_hq32_hkv8_d128_causal":
        VarlenWorkload("llama3_8b_varlen_prefill_bf16_32seq_len128to8192_hq32_hkv8_d128_causal",
                       32, 128, 8192, 32, 8, 128, True),
}


def make_varlen(seqlens_q, seqlens_k, Hq: int, Hkv: int, D: int, seed: int = 0,
                dtype: str = "bf16"):
    """Draw a packed variable-length problem on the CPU: q [sum Tq, Hq, D],
    k and v [sum Tk, Hkv, D], iid N(0, 1) rounded to bf16 (or fp16), and the int32
    offsets cu_seqlens_q, cu_seqlens_k [B + 1] (sequence b at rows cu[b] ..
    cu[b+1]-1)."""
    g = torch.Generator().manual_seed(int(seed))
    lq = [int(x) for x in seqlens_q]
    lk = [int(x) for x in seqlens_k]
    if len(lq) != len(lk):
        raise ValueError("seqlens_q and seqlens_k differ in length")
    tq, tk = sum(lq), sum(lk)
    td = torch_dtype(dtype)
    q = torch.randn(tq, Hq, D, generator=g, dtype=torch.float32).to(td)
    k = torch.randn(tk, Hkv, D, generator=g, dtype=torch.float32).to(td)
    v = torch.randn(tk, Hkv, D, generator=g, dtype=torch.float32).to(td)
    cq = torch.tensor([0] + lq, dtype=torch.int64).cumsum(0).to(torch.int32)
    ck = torch.tensor([0] + lk, dtype=torch.int64).cumsum(0).to(torch.int32)
    return q, k, v, cq, ck


def make_varlen_workload(w: VarlenWorkload, seed: int = 0):
    L = w.seqlens()
    return make_varlen(L, L, w.Hq, w.Hkv, w.D, seed)
