"""The bench's FLOP and byte formulas against the figures the pages print."""
import oracle_pins

from transformer_attention_fwd_gb300.inputs import WORKLOADS, Workload


def test_kv_cache_bytes_match_page_table():
    """"3.3 Self-Attention机制深入理解" §9.4: per-token KV bytes and 4096-token
    totals for 32/8/1 KV heads at head_dim 128, fp16 (2 bytes)."""
    for _, hkv, per_tok, per_4096 in oracle_pins.read_golden("kv_cache_and_flops.txt")[:3]:
        hkv, per_tok, per_4096 = int(hkv), int(per_tok), int(per_4096)
        w = Workload("kv", 1, 32, hkv, 1, 4096, 128, False, "bf16")
        kv_bytes = w.io_bytes() - 2 * (w.B * w.Hq * w.Tq * w.D * 2) - w.B * w.Hq * w.Tq * 4
        assert kv_bytes == per_4096
        assert kv_bytes // 4096 == per_tok


def test_attention_flops_match_page_table():
    """§11.1: QK^T and SV each cost 2 N^2 d; non-causal metric = 4 N^2 d."""
    for row in oracle_pins.read_golden("kv_cache_and_flops.txt"):
        if row[0] != "flops":
            continue
        n, d, f = int(row[1]), int(row[2]), int(row[3])
        w = Workload("f", 1, 1, 1, n, n, d, False, "bf16")
        assert w.flops == f
        assert Workload("f", 1, 1, 1, n, n, d, True, "bf16").flops == f / 2


def test_score_matrix_size_matches_page():
    """"第 11 章 · Attention 入门" §11.4: one fp32 T x T score matrix is 16 MiB at
    T = 2048 and 256 MiB at T = 8192 -- the buffer the tiled kernels avoid."""
    for row in oracle_pins.read_golden("kv_cache_and_flops.txt"):
        if row[0] == "smatrix":
            assert int(row[1]) ** 2 * 4 == int(row[2])


def test_named_workloads():
    w = WORKLOADS["llama3_8b_prefill_bf16_b1_hq32_hkv8_t8192_d128_causal"]
    assert w.flops == 4 * 32 * 8192 * 8192 * 128 / 2
    d = WORKLOADS["gqa_decode_bf16_b64_hq32_hkv8_tk4096_d128"]
    assert d.io_bytes() == 2 * 64 * 8 * 4096 * 128 * 2 + 2 * 64 * 32 * 128 * 2 + 64 * 32 * 4
