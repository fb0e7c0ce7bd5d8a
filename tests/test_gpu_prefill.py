"""CUDA prefill against the fp64 oracle, element by element (relative L2
over all outputs): <= 1e-4 for fp32 inputs, <= 1e-2 for bf16 inputs."""
import zlib

import pytest
import torch

from hybrid_gated_linear_attn_b300 import LizardState, lizard_attn_prefill, lizard_check_device_status
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs, rel_l2
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built, gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(inp, w, tol=None, state=True):
    y_gpu, st = gpu_prefill(inp, w, with_state=state)
    y_ref, S_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], w, state=True)
    tol = tol or TOL[inp["q"].dtype]
    err = rel_l2(y_gpu, y_ref)
    assert err <= tol, f"rel L2 {err:.3e} > {tol}"
    assert torch.isfinite(y_gpu.float()).all()
    if state:
        errS = rel_l2(st.S.cpu(), S_ref)
        assert errS <= tol, f"final state rel L2 {errS:.3e}"
        L, wv = inp["q"].shape[2], st.w
        assert torch.all(st.pos.cpu() == L)
        for p in range(max(0, L - wv), L):
            assert torch.equal(st.ring_k[:, :, p % wv].cpu(), inp["k"][:, :, p])
            assert torch.equal(st.ring_v[:, :, p % wv].cpu(), inp["v"][:, :, p])
    return err


def test_tiny_f32_workload():
    """B1 H2 L256 d64 fp32, w16 m4 alpha 0.5, seed 0 -- the whole output."""
    wl = WORKLOADS["tiny_f32"]
    _check(prefill_inputs(wl), wl.w)


CASES = [
    # name, dtype, B, H, L, d, w, m, g_mean, g_std, alpha
    ("ragged_tail", "bf16", 1, 3, 200, 128, 64, 4, 3.0, 1.0, 1.0),
    ("L_below_w", "bf16", 2, 2, 40, 128, 64, 4, 3.0, 1.0, 1.0),
    ("single_token", "bf16", 2, 2, 1, 128, 16, 4, 3.0, 1.0, 0.5),
    ("no_meta", "f32", 1, 2, 130, 64, 16, 0, 3.0, 1.0, 0.5),
    ("window_one", "f32", 1, 2, 97, 64, 1, 2, 3.0, 1.0, 0.7),
    ("max_window_max_meta", "bf16", 1, 2, 600, 128, 128, 16, 3.0, 1.0, 1.0),
    ("strong_decay", "bf16", 1, 4, 512, 128, 128, 8, 0.0, 2.0, 0.5),
    ("very_strong_decay", "f32", 1, 2, 300, 64, 32, 4, -6.0, 3.0, 1.0),
    ("open_gates", "f32", 1, 2, 200, 64, 16, 4, 12.0, 0.5, 1.0),
    ("d64_bf16", "bf16", 2, 3, 257, 64, 64, 4, 3.0, 1.0, 1.0),
    ("more_units_than_sms", "bf16", 5, 32, 70, 128, 64, 4, 3.0, 1.0, 1.0),
    # tensor-core path edge cases (bf16, d = 128)
    ("extreme_decay_exact_intra", "bf16", 1, 2, 300, 128, 64, 4, -8.0, 4.0, 1.0),
    ("mixed_decay", "bf16", 1, 3, 520, 128, 32, 4, -1.0, 3.0, 0.8),
    ("window_one_bf16", "bf16", 1, 2, 150, 128, 1, 3, 3.0, 1.0, 1.0),
    ("window_65", "bf16", 1, 2, 333, 128, 65, 4, 3.0, 1.0, 1.0),
    ("window_66", "bf16", 1, 2, 333, 128, 66, 4, 3.0, 1.0, 1.0),
    ("one_chunk_exact", "bf16", 2, 2, 64, 128, 64, 4, 3.0, 1.0, 1.0),
    ("alpha_zero", "bf16", 1, 2, 190, 128, 64, 4, 3.0, 1.0, 0.0),
    # few (batch, head) units and long prompts: the prompt runs as sequence
    # segments after a pre-pass for the segments' start states
    ("segments_2", "bf16", 1, 2, 1000, 128, 64, 4, 3.0, 1.0, 1.0),
    ("segments_5_ragged", "bf16", 1, 2, 3000, 128, 48, 4, 3.0, 1.0, 0.7),
    ("segments_strong_decay", "bf16", 1, 2, 2000, 128, 64, 4, 0.0, 2.0, 0.5),
    ("segments_exact_intra", "bf16", 1, 1, 1500, 128, 32, 2, -8.0, 4.0, 1.0),
    ("segments_window_one", "bf16", 1, 2, 1200, 128, 1, 3, 3.0, 1.0, 1.0),
    ("segments_open_gates_no_meta", "bf16", 1, 1, 2500, 128, 64, 0, 12.0, 0.5, 1.0),
    # windows above 65 (three-chunk band) as sequence segments
    ("segments_w100", "bf16", 1, 2, 2000, 128, 100, 4, 3.0, 1.0, 1.0),
    ("segments_w128_strong_decay", "bf16", 1, 2, 2100, 128, 128, 8, 0.0, 2.0, 0.5),
    ("segments_w66_exact_intra", "bf16", 1, 1, 1500, 128, 66, 2, -8.0, 4.0, 1.0),
    # windows 66..128: two earlier band chunks (small prompts, one segment)
    ("w100_single_token", "bf16", 2, 2, 1, 128, 100, 4, 3.0, 1.0, 1.0),
    ("w128_L_below_w", "bf16", 2, 2, 40, 128, 128, 4, 3.0, 1.0, 1.0),
    ("w128_two_chunks", "bf16", 1, 3, 128, 128, 128, 8, 3.0, 1.0, 0.5),
    ("w97_ragged_no_meta", "bf16", 1, 2, 333, 128, 97, 0, 3.0, 1.0, 1.0),
    ("w128_alpha_zero_open_gates", "bf16", 1, 2, 300, 128, 128, 4, 12.0, 0.5, 0.0),
    ("w120_more_units_than_sms", "bf16", 5, 32, 70, 128, 120, 4, 3.0, 1.0, 1.0),
    # w = 64 from the empty state (the instance without the masked
    # selection: the first chunk's missing earlier chunk scores as -inf)
    ("w64_single_token", "bf16", 2, 2, 1, 128, 64, 4, 3.0, 1.0, 1.0),
    ("w64_two_chunks_no_meta", "bf16", 1, 2, 128, 128, 64, 0, 3.0, 1.0, 0.7),
    ("w64_ragged_max_meta", "bf16", 1, 2, 333, 128, 64, 16, 0.0, 2.0, 1.0),
    # head dim 64 on the tensor-core pipeline (tiles zero-padded to 128)
    ("d64_window_one", "bf16", 1, 2, 150, 64, 1, 3, 3.0, 1.0, 1.0),
    ("d64_window_65", "bf16", 1, 2, 333, 64, 65, 4, 3.0, 1.0, 1.0),
    ("d64_extreme_decay_exact_intra", "bf16", 1, 2, 300, 64, 64, 4, -8.0, 4.0, 1.0),
    ("d64_mixed_decay", "bf16", 1, 3, 520, 64, 32, 4, -1.0, 3.0, 0.8),
    ("d64_open_gates_no_meta", "bf16", 1, 2, 200, 64, 48, 0, 12.0, 0.5, 1.0),
    ("d64_max_meta", "bf16", 1, 2, 300, 64, 64, 16, 3.0, 1.0, 1.0),
    ("d64_single_token", "bf16", 2, 2, 1, 64, 16, 4, 3.0, 1.0, 0.5),
    ("d64_L_below_w", "bf16", 2, 2, 40, 64, 64, 4, 3.0, 1.0, 1.0),
    ("d64_alpha_zero", "bf16", 1, 2, 190, 64, 64, 4, 3.0, 1.0, 0.0),
    ("d64_long_prompt_few_units", "bf16", 1, 2, 3000, 64, 64, 4, 3.0, 1.0, 0.7),
    ("d64_more_units_than_sms", "bf16", 5, 32, 70, 64, 64, 4, 3.0, 1.0, 1.0),
    # head dim 64 with two earlier band chunks (windows 66..128)
    ("d64_w100", "bf16", 1, 2, 300, 64, 100, 4, 3.0, 1.0, 1.0),
    ("d64_w128_max_meta_strong_decay", "bf16", 1, 2, 333, 64, 128, 16, 0.0, 2.0, 0.5),
    ("d64_w66_exact_intra", "bf16", 1, 2, 300, 64, 66, 4, -8.0, 4.0, 1.0),
    ("d64_w120_L_below_w", "bf16", 2, 2, 40, 64, 120, 4, 3.0, 1.0, 1.0),
    # head dim 256 on the CUDA cores (four value slices per unit, 32-token chunks)
    ("d256_bf16_ragged", "bf16", 2, 2, 150, 256, 64, 4, 3.0, 1.0, 1.0),
    ("d256_f32_w128_max_meta", "f32", 1, 2, 170, 256, 128, 16, 0.0, 2.0, 0.5),
    ("d256_f32_window_one", "f32", 1, 2, 70, 256, 1, 2, 3.0, 1.0, 0.7),
    ("d256_bf16_single_token", "bf16", 2, 2, 1, 256, 48, 4, 3.0, 1.0, 1.0),
    ("d256_bf16_strong_decay_no_meta", "bf16", 1, 3, 100, 256, 33, 0, -6.0, 3.0, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_small_cases(case):
    name, dt, Bn, H, L, d, w, m, gm, gs, alpha = case
    wl = WORKLOADS["llama3_8b"].replace(B=Bn, H=H, L=L, dk=d, dv=d, w=w, m=m, g_mean=gm, g_std=gs,
                                       alpha=alpha, dtype=dt, seed=zlib.crc32(name.encode()) % 1000)
    _check(prefill_inputs(wl), w)


def test_empty_sequence_writes_empty_state():
    wl = WORKLOADS["llama3_8b"].replace(B=1, H=2, L=0)
    inp = prefill_inputs(wl)
    y, st = gpu_prefill(inp, wl.w)
    assert y.numel() == 0
    assert torch.all(st.S.cpu() == 0) and torch.all(st.pos.cpu() == 0)


def _full_size(wl_name):
    """One launch at the workload's full size; the oracle (one thread per
    unit) on every (batch, head) unit: y and the final state over all
    elements."""
    wl = WORKLOADS[wl_name]
    inp = prefill_inputs(wl)
    y_gpu, st = gpu_prefill(inp, wl.w)
    y_ref, S_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], wl.w, state=True)
    tol = TOL[inp["q"].dtype]
    assert torch.isfinite(y_gpu.float()).all()
    err = rel_l2(y_gpu, y_ref)
    assert err <= tol, f"{wl_name}: y rel L2 {err:.3e}"
    errS = rel_l2(st.S.cpu(), S_ref)
    assert errS <= tol, f"{wl_name}: final state rel L2 {errS:.3e}"
    # per unit too: no single head may hide behind the others
    per_unit = [rel_l2(y_gpu[b, h], y_ref[b, h]) for b in range(wl.B) for h in range(wl.H)]
    assert max(per_unit) <= tol, f"{wl_name}: worst unit rel L2 {max(per_unit):.3e}"


def test_llama3_8b_full_size_all_units():
    """B4 H32 L4096 d128 bf16 in one launch; all 128 units against the oracle."""
    _full_size("llama3_8b")


def test_d64_full_size_all_units():
    """B4 H32 L4096 d64 bf16 (the tensor-core pipeline on zero-padded
    tiles) in one launch; all 128 units against the oracle."""
    _full_size("d64")


def test_decay_stress_full_size_all_units():
    """B2 H32 L8192 d128 bf16, g ~ N(0, 2): cumulative decay far below fp32
    range; all 64 units against the oracle."""
    _full_size("decay_stress")


def test_calls_on_batch_slices_with_state_views():
    """One call per sequence, each on a LizardState.batch view, writes the
    same outputs and state rows as the oracle run over the whole batch."""
    wl = WORKLOADS["llama3_8b"].replace(B=3, H=2, L=700, seed=77)
    inp = prefill_inputs(wl)
    q, k, v, g, mu = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu"))
    st = LizardState(wl.B, wl.H, wl.dk, wl.dv, wl.w, dtype=q.dtype)
    y = torch.empty_like(v)
    for b in range(wl.B):
        lizard_attn_prefill(q[b:b + 1], k[b:b + 1], v[b:b + 1], g[b:b + 1], mu, wl.alpha, wl.w, y=y[b:b + 1],
                            state=st.batch(b, b + 1))
    torch.cuda.synchronize()
    lizard_check_device_status()
    y_ref, S_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], wl.w, state=True)
    assert rel_l2(y.cpu(), y_ref) <= TOL[q.dtype]
    assert rel_l2(st.S.cpu(), S_ref) <= TOL[q.dtype]
    assert torch.all(st.pos.cpu() == wl.L)
    for p in range(wl.L - wl.w, wl.L):
        assert torch.equal(st.ring_k[:, :, p % wl.w].cpu(), inp["k"][:, :, p])
