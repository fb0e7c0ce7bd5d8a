"""The library's scratch pool: memory a call needed for temporary data stays
reserved for later calls until lizard_scratch_trim hands it back."""
import pytest
import torch

from hybrid_gated_linear_attn_b300 import (lizard_attn_backward, lizard_check_device_status, lizard_scratch_reserved,
                                           lizard_scratch_trim)
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs
from tests.gpu_helpers import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_trim_returns_the_scratch_of_a_backward():
    wl = WORKLOADS["llama3_8b"].replace(B=4, H=16, L=2048)  # 64 units x 32 chunks: about 190 MB of scratch
    inp = prefill_inputs(wl)
    q, k, v, g, mu = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu"))
    dy = torch.randn_like(q)
    torch.cuda.synchronize()
    lizard_scratch_trim(0)
    torch.cuda.empty_cache()
    free0, _ = torch.cuda.mem_get_info()
    assert lizard_scratch_reserved() == 0
    grads = lizard_attn_backward(q, k, v, g, mu, wl.alpha, wl.w, dy)
    lizard_check_device_status()  # synchronises the stream
    del grads
    held = lizard_scratch_reserved()
    # chunk states and state gradients (bf16), q * dq (fp32): well above 100 MB
    assert held >= 100 << 20, held
    free1, _ = torch.cuda.mem_get_info()
    assert free1 <= free0 - held + (64 << 20)
    # a second call maps nothing new
    grads = lizard_attn_backward(q, k, v, g, mu, wl.alpha, wl.w, dy)
    lizard_check_device_status()
    del grads
    assert lizard_scratch_reserved() == held
    lizard_scratch_trim(0)
    assert lizard_scratch_reserved() == 0
    torch.cuda.empty_cache()  # the gradients the calls returned were dropped
    free2, _ = torch.cuda.mem_get_info()
    assert free2 >= free0 - (64 << 20), (free0, free2)
