"""Gate projection (lizard_gate_projection) against the fp64 oracle.

g = x W_gamma^T in the operator's head-major layout; bf16 output, compared
element by element (relative L2 <= 1e-2, the bf16 tolerance).
"""
import pytest
import torch

from hybrid_gated_linear_attn_b300 import lizard_attn_prefill, lizard_gate_projection
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, gate_projection_inputs, prefill_inputs, rel_l2
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


CASES = [
    # B, L, dmodel, H
    (1, 128, 64, 1),      # one tile, one K slice
    (2, 300, 256, 3),     # ragged token blocks across the batch boundary
    (1, 130, 200, 2),     # K not a multiple of the 64-wide slice
    (3, 77, 512, 4),
    (1, 1, 1024, 2),      # a single token
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}_L{c[1]}_dm{c[2]}_H{c[3]}" for c in CASES])
def test_gate_projection_small(case):
    B, L, dm, H = case
    inp = gate_projection_inputs(B, L, dm, H, 128, seed=sum(case))
    g = lizard_gate_projection(inp["x"].cuda(), inp["W"].cuda(), H)
    torch.cuda.synchronize()
    ref = O.gate_projection(inp["x"], inp["W"], H)
    err = rel_l2(g.cpu(), ref)
    assert err <= TOL[torch.bfloat16], f"rel L2 {err:.3e}"


def test_gate_projection_llama3_8b_sampled_rows():
    """B4 L4096 dmodel 4096, H32 x 128: one launch; the oracle on 96 sampled
    tokens (all heads)."""
    B, L, dm, H = 4, 4096, 4096, 32
    inp = gate_projection_inputs(B, L, dm, H, 128)
    g = lizard_gate_projection(inp["x"].cuda(), inp["W"].cuda(), H)
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(7)
    bs = torch.randint(0, B, (96,), generator=gen)
    ts = torch.randint(0, L, (96,), generator=gen)
    xs = inp["x"][bs, ts][:, None, :]                          # [96, 1, dm]
    ref = O.gate_projection(xs, inp["W"], H)[:, :, 0, :]       # [96, H, 128]
    got = g.cpu()[bs, :, ts, :]                                # [96, H, 128]
    err = rel_l2(got, ref)
    assert err <= TOL[torch.bfloat16], f"rel L2 {err:.3e}"


def test_projection_feeds_the_operator():
    """x -> g (this kernel) -> prefill equals the prefill of the oracle's g
    (same bf16 bits when the kernel's g matches)."""
    wl = WORKLOADS["llama3_8b"].replace(B=1, H=2, L=200)
    inp = prefill_inputs(wl)
    proj = gate_projection_inputs(1, 200, 256, 2, 128, seed=3)
    g = lizard_gate_projection(proj["x"].cuda(), proj["W"].cuda(), 2)
    q, k, v, mu = (inp[n].cuda() for n in ("q", "k", "v", "mu"))
    y = lizard_attn_prefill(q, k, v, g, mu, wl.alpha, wl.w)
    torch.cuda.synchronize()
    g_ref = O.gate_projection(proj["x"], proj["W"], 2).to(torch.bfloat16)
    y_ref = O.forward(inp["q"], inp["k"], inp["v"], g_ref, inp["mu"], wl.alpha, wl.w)
    assert rel_l2(y.cpu(), y_ref) <= TOL[torch.bfloat16]
