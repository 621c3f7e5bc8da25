"""fp32 I/O parity against the float64 oracle (tolerance 1e-5)."""
import pytest

import oracle
from gpu_util import TOL_LSE_F32, TOL_O_F32, attn, check_status, compare, to_dev
from transformer_attention_fwd_gb300.inputs import WORKLOADS, make_qkv, make_workload

pytestmark = pytest.mark.gpu

F32_NAMED = ["sdpa_f32_b1_h1_t128_d64_causal", "sdpa_f32_b1_h4_t128_d64_causal",
             "sdpa_f32_b1_h4_t128_d64_noncausal"]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", F32_NAMED)
def test_named_fp32_workloads(name, seed):
    a = attn()
    w = WORKLOADS[name]
    q, k, v = make_workload(w, seed)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=w.causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, w.causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_F32, TOL_LSE_F32, name)


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tk,D,causal", [
    (1, 1, 1, 1, 1, 64, True), (2, 3, 1, 7, 7, 64, True), (1, 2, 2, 33, 90, 128, True),
    (1, 4, 2, 130, 130, 128, False), (2, 8, 8, 5, 300, 64, False), (1, 2, 1, 17, 17, 64, False),
])
def test_fp32_edge_shapes(B, Hq, Hkv, Tq, Tk, D, causal):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, D, "f32", seed=Tq + Tk)
    o, lse = a.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_status(a)
    o_ref, lse_ref = oracle.attention_f64(q, k, v, causal)
    compare(o, lse, o_ref, lse_ref, TOL_O_F32, TOL_LSE_F32)
