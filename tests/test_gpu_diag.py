"""Self-tests of the hardware building blocks (tensor-core tile products,
bounded pipeline waits), run before the attention parity tests."""
import pytest
import torch

from gpu_util import attn, check_status

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
def test_mma_tile_products(D):
    a_ = attn()
    g = torch.Generator().manual_seed(D)
    A = torch.randn(128, D, generator=g).to(torch.bfloat16)
    Bm = torch.randn(128, D, generator=g).to(torch.bfloat16)
    V = torch.randn(128, D, generator=g).to(torch.bfloat16)
    s, o = a_.diag_mma_tile(A.cuda(), Bm.cuda(), V.cuda())
    check_status(a_)
    s = s.cpu().double()
    s_ref = A.double() @ Bm.double().T
    err_s = (s - s_ref).abs().max().item()
    assert err_s <= 1e-3 * max(1.0, s_ref.abs().max().item()), f"S tile error {err_s}"
    # O = bf16(S) . V, with P taken from the kernel's own S (rounded as the kernel rounds).
    p = s.float().to(torch.bfloat16).double()
    o_ref = p @ V.double()
    err_o = (o.cpu().double() - o_ref).abs().max().item()
    assert err_o <= 1e-3 * max(1.0, o_ref.abs().max().item()), f"O tile error {err_o}"


def test_bounded_wait_reports_timeout_and_context_survives():
    a_ = attn()
    a_.diag_wait_timeout(1_000_000)  # 1 ms limit on a barrier nobody signals
    assert a_.device_status() == a_.ATTN_ERR_TIMEOUT
    assert "timed out" in a_.last_error()
    assert a_.device_status() == a_.ATTN_OK  # cleared by the read
    x = torch.ones(1024, device="cuda")
    assert float((x * 2).sum()) == 2048.0  # the context is still usable
