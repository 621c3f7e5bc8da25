"""attn_fwd_host: the same computation as attn_fwd on host buffers, with the
copies pipelined against the compute over chunks of (b, hkv) pairs.  Each
chunk is attn_fwd on a sub-problem, so the outputs equal attn_fwd's bit for
bit."""
import pytest
import torch

from gpu_util import attn, check_status
from transformer_attention_fwd_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def _chunk_bounds(units, max_chunks=5, edge_div=2):
    """The library's chunking of (b, hkv) pairs: up to five chunks, the first
    and last holding units // (2 * chunks) pairs (at least one)."""
    chunks = min(units, max_chunks)
    if chunks < 3:
        return [c * units // chunks for c in range(chunks + 1)]
    edge = max(1, units // (edge_div * chunks))
    mid, nm = units - 2 * edge, chunks - 2
    return [0, edge] + [edge + c * mid // nm for c in range(1, nm + 1)] + [units]


@pytest.mark.parametrize("dtype,B,Hq,Hkv,Tq,Tk,D,causal", [
    ("bf16", 2, 8, 2, 700, 700, 128, True),    # 4 pairs: 4 chunks of one
    ("bf16", 1, 32, 8, 1, 4096, 128, False),   # decode, 8 pairs
    ("f16", 3, 6, 3, 300, 500, 64, True),      # 9 pairs into 5 chunks of 1, 2, 2, 3, 1
    ("f32", 1, 4, 4, 128, 128, 64, True),      # the CUDA-core path
])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_call_equals_device_call(dtype, B, Hq, Hkv, Tq, Tk, D, causal, pinned):
    a = attn()
    q, k, v = make_qkv(B, Hq, Hkv, Tq, Tk, D, dtype, seed=131)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_h, l_h = a.attn_fwd_host(q, k, v, causal=causal)
    torch.cuda.synchronize()
    check_status(a)
    # The device call on each chunk's sub-problem, for a bit-exact reference.
    units, g = B * Hkv, Hq // Hkv
    bound = _chunk_bounds(units)
    qd = q.cuda().reshape(units, g, Tq, D)
    kd, vd = k.cuda().reshape(units, 1, Tk, D), v.cuda().reshape(units, 1, Tk, D)
    o_ref = torch.empty_like(qd)
    l_ref = torch.empty((units, g, Tq), dtype=torch.float32, device="cuda")
    for u0, u1 in zip(bound[:-1], bound[1:]):
        a.attn_fwd(qd[u0:u1], kd[u0:u1], vd[u0:u1], causal=causal, out=o_ref[u0:u1],
                   lse=l_ref[u0:u1])
    check_status(a)
    assert not o_h.is_cuda and o_h.dtype == q.dtype
    assert torch.equal(o_h.reshape(units, g, Tq, D), o_ref.cpu())
    assert torch.equal(l_h.reshape(units, g, Tq), l_ref.cpu())


def test_host_call_without_lse_and_in_a_graph():
    a = attn()
    q, k, v = (x.pin_memory() for x in make_qkv(2, 8, 4, 256, 256, 128, "bf16", seed=132))
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    a.attn_fwd_host(q, k, v, causal=True, out=o, want_lse=False)
    torch.cuda.synchronize()
    ref = o.clone()
    o.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.attn_fwd_host(q, k, v, causal=True, out=o, want_lse=False)
    g.replay()
    torch.cuda.synchronize()
    check_status(a)
    assert torch.equal(o, ref)
