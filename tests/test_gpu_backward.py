"""CUDA backward (lizard_attn_backward) against the fp64 oracle's backward.

Every gradient -- dq, dk, dv, dg, d meta_k, d alpha -- is compared element
by element (relative L2 over the whole tensor): <= 1e-4 for fp32 inputs,
<= 1e-2 for bf16 inputs (whose gradients are rounded to bf16 once).
"""
import zlib

import pytest
import torch

from hybrid_gated_linear_attn_b300 import lizard_attn_backward
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs, rel_l2
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _case_inputs(name, dt, Bn, H, L, d, w, m, gm=3.0, gs=1.0, alpha=1.0):
    seed = zlib.crc32(name.encode()) % 1000
    wl = WORKLOADS["llama3_8b"].replace(B=Bn, H=H, L=L, dk=d, dv=d, w=w, m=m, g_mean=gm, g_std=gs,
                                       alpha=alpha, dtype=dt, seed=seed)
    inp = prefill_inputs(wl)
    gen = torch.Generator().manual_seed(seed + 7)
    inp["dy"] = torch.randn(Bn, H, L, d, generator=gen).to(inp["q"].dtype)
    return inp


def _gpu_backward(inp, w):
    q, k, v, g, mu, dy = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu", "dy"))
    out = lizard_attn_backward(q, k, v, g, mu if mu.shape[1] > 0 else None, inp["alpha"], w, dy)
    torch.cuda.synchronize()
    return [None if t is None else t.cpu() for t in out]


def _dalpha_error(inp, w, got: float, ref: float) -> float:
    """Error of d alpha = sum_t dy_t . ya_t relative to |d alpha|.  The
    sum has B H L d_v terms of both signs; its rounding errors are
    independent per term, so their natural scale is the L2 norm of the
    terms, ||dy * ya||_2, which is also the typical size of |d alpha| for a
    random dy.  When a seed makes the sum cancel to below 1/20 of that size
    the relative error is measured against that size instead."""
    _, _, ya = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], w, branches=True)
    scale = float((inp["dy"].double() * ya).norm())
    return abs(got - ref) / max(abs(ref), scale / 20.0, 1e-30)


def _check(inp, w):
    dq, dk, dv, dg, dmu, dal = _gpu_backward(inp, w)
    ref = O.backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], w, inp["dy"].double())
    tol = TOL[inp["q"].dtype]
    errs = {}
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg)):
        assert torch.isfinite(got.float()).all(), name
        if float(ref[name].norm()) > 0:
            errs[name] = rel_l2(got, ref[name])
        else:
            # dg is exactly 0 when every token's gate only scales the empty
            # state (a single token): it is q*dq - k*dk, two equal terms, and
            # fp32 leaves a rounding residue on the scale of those terms.
            scale = float((inp["q"].double() * ref["dq"]).norm())
            errs[name] = float(got.double().norm()) / max(scale, 1e-30)
    if inp["mu"].shape[1] > 0:
        if float(ref["dmu"].norm()) > 0:
            errs["dmu"] = rel_l2(dmu, ref["dmu"])
        else:  # alpha = 0: the sinks get no gradient at all
            errs["dmu"] = 0.0 if float(dmu.abs().max()) == 0.0 else float("inf")
    errs["dalpha"] = _dalpha_error(inp, w, float(dal), float(ref["dalpha"]))
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"rel L2 above {tol}: {bad} (all: {errs})"
    return errs


CASES = [
    # name, dtype, B, H, L, d, w, m, g_mean, g_std, alpha
    ("f32_d64", "f32", 1, 2, 70, 64, 16, 4, 3.0, 1.0, 0.7),
    ("f32_d128", "f32", 1, 2, 100, 128, 64, 4, 3.0, 1.0, 1.0),
    ("f32_long", "f32", 1, 1, 1000, 64, 32, 3, 2.0, 1.5, 0.9),
    ("bf16_d128_w64", "bf16", 2, 2, 200, 128, 64, 4, 3.0, 1.0, 1.0),
    ("bf16_L_below_w", "bf16", 1, 2, 20, 128, 64, 4, 3.0, 1.0, 1.0),
    ("f32_single_token", "f32", 1, 1, 1, 64, 16, 2, 3.0, 1.0, 0.5),
    ("f32_no_meta", "f32", 1, 2, 90, 64, 16, 0, 3.0, 1.0, 0.5),
    ("f32_window_one", "f32", 1, 2, 77, 64, 1, 2, 3.0, 1.0, 0.7),
    ("bf16_max_window_max_meta", "bf16", 1, 2, 300, 128, 128, 16, 3.0, 1.0, 1.0),
    ("f32_strong_decay", "f32", 1, 2, 150, 64, 32, 4, -8.0, 4.0, 1.0),
    ("f32_open_gates", "f32", 1, 2, 130, 64, 16, 4, 12.0, 0.5, 1.0),
    ("f32_alpha_zero", "f32", 1, 2, 80, 64, 16, 4, 3.0, 1.0, 0.0),
    ("bf16_d64_w100", "bf16", 2, 3, 257, 64, 100, 4, 3.0, 1.0, 1.0),
    ("bf16_mixed_decay", "bf16", 1, 3, 333, 128, 48, 4, -1.0, 3.0, 0.8),
    # tensor-core path (bf16, d = 128, w <= 65): chunk boundaries, ragged
    # tails, wide-span chunks on the exact path, windows 1 .. 65
    ("tc_one_chunk", "bf16", 2, 2, 64, 128, 64, 4, 3.0, 1.0, 1.0),
    ("tc_chunk_plus_one", "bf16", 1, 2, 65, 128, 64, 4, 3.0, 1.0, 1.0),
    ("tc_single_token", "bf16", 1, 2, 1, 128, 64, 4, 3.0, 1.0, 1.0),
    ("tc_window_one", "bf16", 1, 2, 190, 128, 1, 3, 3.0, 1.0, 1.0),
    ("tc_window_33", "bf16", 1, 2, 300, 128, 33, 2, 3.0, 1.0, 0.6),
    ("tc_window_65_max_meta", "bf16", 1, 2, 260, 128, 65, 16, 3.0, 1.0, 1.0),
    ("tc_no_meta", "bf16", 1, 2, 200, 128, 64, 0, 3.0, 1.0, 1.0),
    ("tc_alpha_zero", "bf16", 1, 2, 150, 128, 64, 4, 3.0, 1.0, 0.0),
    ("tc_wide_span_exact", "bf16", 1, 2, 300, 128, 64, 4, -8.0, 4.0, 1.0),
    ("tc_strong_decay", "bf16", 1, 2, 256, 128, 64, 8, 0.0, 2.0, 0.5),
    ("tc_open_gates", "bf16", 1, 2, 200, 128, 32, 4, 12.0, 0.5, 1.0),
    ("tc_many_units", "bf16", 3, 8, 130, 128, 64, 4, 3.0, 1.0, 1.0),
    # tensor-core path with head dim 64 (tiles zero-padded to 128)
    ("tc_d64_w64", "bf16", 2, 2, 200, 64, 64, 4, 3.0, 1.0, 1.0),
    ("tc_d64_one_chunk", "bf16", 2, 2, 64, 64, 64, 4, 3.0, 1.0, 1.0),
    ("tc_d64_single_token", "bf16", 1, 2, 1, 64, 64, 4, 3.0, 1.0, 1.0),
    ("tc_d64_window_one", "bf16", 1, 2, 190, 64, 1, 3, 3.0, 1.0, 1.0),
    ("tc_d64_wide_span_exact", "bf16", 1, 2, 300, 64, 64, 4, -8.0, 4.0, 1.0),
    ("tc_d64_no_meta", "bf16", 1, 2, 200, 64, 32, 0, 3.0, 1.0, 1.0),
    ("tc_d64_window_65_max_meta", "bf16", 1, 2, 260, 64, 65, 16, 3.0, 1.0, 1.0),
    ("tc_d64_alpha_zero", "bf16", 1, 2, 150, 64, 64, 4, 3.0, 1.0, 0.0),
    ("tc_d64_open_gates", "bf16", 1, 2, 200, 64, 32, 4, 12.0, 0.5, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_small_cases(case):
    name, dt, Bn, H, L, d, w, m, gm, gs, alpha = case
    _check(_case_inputs(name, dt, Bn, H, L, d, w, m, gm, gs, alpha), w)


def test_empty_sequence_gives_zero_parameter_gradients():
    inp = _case_inputs("empty", "bf16", 1, 2, 0, 128, 64, 4)
    dq, dk, dv, dg, dmu, dal = _gpu_backward(inp, 64)
    assert dq.numel() == 0 and float(dal) == 0.0 and torch.all(dmu == 0)


def _full_size(wl_name, seed):
    """One launch at the workload's full size; the oracle backward on every
    (batch, head) unit (one thread per unit); every gradient compared over
    all elements."""
    wl = WORKLOADS[wl_name]
    inp = prefill_inputs(wl)
    gen = torch.Generator().manual_seed(seed)
    inp["dy"] = torch.randn(wl.B, wl.H, wl.L, wl.dv, generator=gen).to(inp["q"].dtype)
    dq, dk, dv, dg, dmu, dal = _gpu_backward(inp, wl.w)
    ref = O.backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], wl.alpha, wl.w, inp["dy"].double())
    tol = TOL[torch.bfloat16]
    errs = {n: rel_l2(got, ref[n]) for n, got in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg), ("dmu", dmu))}
    errs["dalpha"] = _dalpha_error(inp, wl.w, float(dal), float(ref["dalpha"]))
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"{wl_name}: above {tol}: {bad} (all: {errs})"


def test_llama3_8b_full_size_all_units():
    """B4 H32 L4096 d128 bf16 (tensor-core path), all 128 units."""
    _full_size("llama3_8b", 99)


def test_decay_stress_full_size_all_units():
    """B2 H32 L8192 d128 bf16, g ~ N(0, 2), w128 m8 alpha 0.5 (w > 65: the
    exact CUDA-core path), all 64 units."""
    _full_size("decay_stress", 98)


def test_d64_full_size_all_units():
    """B4 H32 L4096 d64 bf16 (the tensor-core path on zero-padded tiles),
    all 128 units."""
    _full_size("d64", 97)
