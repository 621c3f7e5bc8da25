"""Every entry point can be captured into a CUDA graph and replayed: the
launches, the stream-ordered workspace allocations and the scheduling kernels
all live on the caller's stream, so a replay recomputes exactly what an eager
call computes.  A graph is how a caller removes the per-call launch cost."""
import pytest
import torch

from gpu_util import attn, check_status
from transformer_attention_fwd_gb300.inputs import make_paged, make_qkv, make_varlen

pytestmark = pytest.mark.gpu


def _replay_equals_eager(fn, outs):
    """fn() writes into the tensors of `outs`; eager result vs 3 replays."""
    a = attn()
    fn()  # eager (also sets kernel attributes outside the capture)
    torch.cuda.synchronize()
    check_status(a)
    ref = [o.clone() for o in outs]
    for o in outs:
        o.fill_(0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    for _ in range(3):
        for o in outs:
            o.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        for o, r in zip(outs, ref):
            assert torch.equal(o, r)
    check_status(a)


@pytest.mark.parametrize("dtype,Tq,causal", [("bf16", 700, True), ("bf16", 1, False),
                                             ("f16", 300, False), ("f16", 1, False)])
def test_attn_fwd_in_a_graph(dtype, Tq, causal):
    a = attn()
    q, k, v = (x.cuda() for x in make_qkv(2, 8, 2, Tq, 900, 128, dtype, seed=121))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    _replay_equals_eager(lambda: a.attn_fwd(q, k, v, causal=causal, out=o, lse=lse), [o, lse])


def test_window_in_a_graph():
    a = attn()
    q, k, v = (x.cuda() for x in make_qkv(1, 8, 2, 600, 600, 64, "bf16", seed=122))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    _replay_equals_eager(lambda: a.attn_fwd_window(q, k, v, 200, out=o, lse=lse), [o, lse])


def test_varlen_in_a_graph():
    a = attn()
    q, k, v, cq, ck = (x.cuda() for x in make_varlen([300, 5, 0, 700], [300, 40, 8, 700],
                                                      8, 2, 128, seed=123))
    o = torch.empty_like(q)
    lse = torch.empty((8, q.shape[0]), dtype=torch.float32, device="cuda")
    _replay_equals_eager(lambda: a.attn_fwd_varlen(q, k, v, cq, ck, True, out=o, lse=lse), [o, lse])


def test_paged_decode_in_a_graph():
    a = attn()
    q, kv, bt, sl = (x.cuda() for x in make_paged(6, 16, 4, 128, 16, [1000, 1, 0, 77, 2048, 500],
                                                  seed=124))
    o = torch.empty_like(q)
    lse = torch.empty((6, 16), dtype=torch.float32, device="cuda")
    _replay_equals_eager(lambda: a.attn_fwd_decode_paged(q, kv, bt, sl, out=o, lse=lse), [o, lse])


def test_split_decode_in_a_graph():
    a = attn()
    q, k, v = (x.cuda() for x in make_qkv(4, 16, 4, 1, 3000, 64, "bf16", seed=125))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    _replay_equals_eager(lambda: a.attn_fwd_decode(q, k, v, num_splits=7, out=o, lse=lse), [o, lse])
