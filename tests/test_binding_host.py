"""Host-side checks of the Python binding's argument checks (no GPU needed):
caller-supplied output buffers must hold exactly what a call writes, since
the kernels write through their pointers and know nothing of their sizes,
and all tensors of a call must sit on one device."""
import pytest
import torch


@pytest.fixture(scope="module")
def a():
    from transformer_attention_fwd_gb300 import build
    build.build()
    from transformer_attention_fwd_gb300 import attn
    return attn


def test_matching_buffer_and_none_pass(a):
    a._check_buffer("out", None, (2, 3), torch.float32, "cpu")
    a._check_buffer("out", torch.empty(2, 3), (2, 3), torch.float32, "cpu")
    # Only the element count matters for the shape: [B, Hq, 1] serves [B, Hq].
    a._check_buffer("lse", torch.empty(4, 8, 1), (4, 8), torch.float32, "cpu")


@pytest.mark.parametrize("buf,msg", [
    (torch.empty(2, 4), "elements"),                     # too large
    (torch.empty(5), "elements"),                        # too small
    (torch.empty(2, 3, dtype=torch.bfloat16), "float32"),
    (torch.empty(3, 2).t(), "contiguous"),
    (torch.empty(2, 3, device="meta"), "on cpu"),
])
def test_mismatched_buffers_rejected(a, buf, msg):
    with pytest.raises(ValueError, match=msg):
        a._check_buffer("out", buf, (2, 3), torch.float32, "cpu")


def test_tensors_on_two_devices_rejected(a):
    a._same_device(q=torch.empty(1), k=torch.empty(1))
    with pytest.raises(ValueError, match="one device"):
        a._same_device(q=torch.empty(1), k=torch.empty(1, device="meta"))


def test_host_call_rejects_a_short_output_before_the_library(a):
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="out must hold"):
        a.attn_fwd_host(q, k, k, out=torch.empty(1, 2, 7, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="lse must hold"):
        a.attn_fwd_host(q, k, k, lse=torch.empty(1, 2, 9))
