"""CUDA decode step against the fp64 oracle's decode step and against the
oracle's prefill of the whole sequence (bf16: rel L2 <= 1e-2)."""
import pytest
import torch

from hybrid_gated_linear_attn_b300 import LizardState, lizard_state_init
from hybrid_gated_linear_attn_b300.inputs import (WORKLOADS, decode_initial_state, decode_step_inputs,
                                                  prefill_inputs, rel_l2, torch_dtype)
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built, gpu_decode_step, gpu_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _gpu_state_from(init: dict, wl) -> LizardState:
    st = LizardState(wl.B, wl.H, wl.dk, wl.dv, wl.w, dtype=init["ring_k"].dtype)
    st.S.copy_(init["S"])
    st.ring_k.copy_(init["ring_k"])
    st.ring_v.copy_(init["ring_v"])
    st.pos.copy_(init["pos"])
    return st


def _run_decode(wl, steps, seq=None):
    init = decode_initial_state(wl)
    st = _gpu_state_from(init, wl)
    seq = list(range(wl.B)) if seq is None else seq
    ost = dict(S=init["S"][seq].double().contiguous(), ring_k=init["ring_k"][seq].contiguous(),
               ring_v=init["ring_v"][seq].contiguous(), pos=init["pos"][seq].clone())
    worst = 0.0
    for s in range(steps):
        inp = decode_step_inputs(wl, s)
        y = gpu_decode_step(inp, init["mu"], wl.alpha, st).cpu()
        sub = {n: inp[n][seq].contiguous() for n in ("q", "k", "v", "g")}
        y_ref = O.decode_step(sub["q"], sub["k"], sub["v"], sub["g"], init["mu"], wl.alpha, ost)
        err = rel_l2(y[seq], y_ref)
        worst = max(worst, err)
        assert err <= TOL[inp["q"].dtype], f"step {s}: rel L2 {err:.3e}"
    errS = rel_l2(st.S.cpu()[seq], ost["S"])
    assert errS <= TOL[torch_dtype(wl.dtype)], f"state rel L2 {errS:.3e}"
    assert torch.all(st.pos.cpu() == init["pos"] + steps)
    for b_local, b in enumerate(seq):
        assert torch.equal(st.ring_k.cpu()[b], ost["ring_k"][b_local])
        assert torch.equal(st.ring_v.cpu()[b], ost["ring_v"][b_local])
    return worst


@pytest.mark.parametrize("d,w,m,hist,dtype", [
    (128, 64, 4, 64, "bf16"),     # full ring
    (128, 64, 4, 10, "bf16"),     # ring still filling (pos < w)
    (64, 16, 0, 40, "f32"),       # no sinks
    (64, 1, 3, 5, "f32"),         # window of one token
    (128, 128, 16, 300, "bf16"),  # largest window and meta count
    (256, 64, 4, 70, "bf16"),     # head dim 256: eight value slices per unit
    (256, 96, 16, 20, "f32"),     # head dim 256 in fp32, ring still filling
])
def test_decode_small(d, w, m, hist, dtype):
    wl = WORKLOADS["decode"].replace(B=3, H=4, dk=d, dv=d, w=w, m=m, L=hist, dtype=dtype)
    _run_decode(wl, steps=2 * w + 3)


def test_decode_from_empty_state():
    wl = WORKLOADS["decode"].replace(B=2, H=3, L=0)
    st = LizardState(wl.B, wl.H, wl.dk, wl.dv, wl.w, dtype=torch.bfloat16)
    lizard_state_init(st)
    torch.cuda.synchronize()
    assert torch.all(st.S.cpu() == 0) and torch.all(st.pos.cpu() == 0)
    init = decode_initial_state(wl)
    ost = dict(S=torch.zeros(wl.B, wl.H, wl.dk, wl.dv, dtype=torch.float64),
               ring_k=torch.zeros_like(init["ring_k"]), ring_v=torch.zeros_like(init["ring_v"]),
               pos=torch.zeros(wl.B, dtype=torch.int64))
    for s in range(5):
        inp = decode_step_inputs(wl, s)
        y = gpu_decode_step(inp, init["mu"], wl.alpha, st).cpu()
        y_ref = O.decode_step(inp["q"], inp["k"], inp["v"], inp["g"], init["mu"], wl.alpha, ost)
        assert rel_l2(y, y_ref) <= 1e-2


def test_decode_workload_full_size_all_sequences():
    """64 sequences x H32 d128 bf16, w64 m4, 1024 steps in one state; the
    oracle follows every sequence for every step (sequences in groups, one
    oracle thread per group), and the final state, ring and pos of all of
    them are compared."""
    import threading
    wl = WORKLOADS["decode"]
    init = decode_initial_state(wl)
    st = _gpu_state_from(init, wl)
    groups = [list(range(i, min(wl.B, i + 4))) for i in range(0, wl.B, 4)]
    ost = [dict(S=init["S"][g].double().contiguous(), ring_k=init["ring_k"][g].contiguous(),
                ring_v=init["ring_v"][g].contiguous(), pos=init["pos"][g].clone()) for g in groups]
    tol = TOL[torch.bfloat16]
    for s in range(wl.decode_steps):
        inp = decode_step_inputs(wl, s)
        y = gpu_decode_step(inp, init["mu"], wl.alpha, st).cpu()
        refs = [None] * len(groups)

        def run(i):
            sub = {n: inp[n][groups[i]].contiguous() for n in ("q", "k", "v", "g")}
            refs[i] = O.decode_step(sub["q"], sub["k"], sub["v"], sub["g"], init["mu"], wl.alpha, ost[i])

        ths = [threading.Thread(target=run, args=(i,)) for i in range(len(groups))]
        for t in ths:
            t.start()
        for t in ths:
            t.join()
        y_ref = torch.cat(refs)
        err = rel_l2(y, y_ref)
        assert err <= tol, f"step {s}: rel L2 {err:.3e}"
    S_ref = torch.cat([o["S"] for o in ost])
    errS = rel_l2(st.S.cpu(), S_ref)
    assert errS <= tol, f"state rel L2 {errS:.3e}"
    assert torch.all(st.pos.cpu() == init["pos"] + wl.decode_steps)
    assert torch.equal(st.ring_k.cpu(), torch.cat([o["ring_k"] for o in ost]))
    assert torch.equal(st.ring_v.cpu(), torch.cat([o["ring_v"] for o in ost]))


@pytest.mark.parametrize("L,w,n", [(100, 64, 9), (20, 64, 70), (130, 16, 5)])
def test_prefill_then_decode_equals_longer_prefill(L, w, n):
    wl = WORKLOADS["llama3_8b"].replace(B=2, H=3, L=L + n, w=w, seed=L)
    inp = prefill_inputs(wl)
    head = {k: (v[:, :, :L].contiguous() if isinstance(v, torch.Tensor) and k != "mu" else v)
            for k, v in inp.items()}
    _, st = gpu_prefill(head, w)
    y_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], w)
    for t in range(L, L + n):
        step = {k: inp[k][:, :, t].contiguous() for k in ("q", "k", "v", "g")}
        y = gpu_decode_step(step, inp["mu"], inp["alpha"], st).cpu()
        err = rel_l2(y, y_ref[:, :, t])
        assert err <= 1e-2, f"t={t}: rel L2 {err:.3e}"


def test_decode_reports_a_position_outside_the_valid_range():
    """A pos outside [0, 2^40) is reported by lizard_check_device_status;
    the other sequences of the same call are still exact and every pos of a
    valid sequence advances by one."""
    from hybrid_gated_linear_attn_b300 import LizardError, lizard_check_device_status
    from hybrid_gated_linear_attn_b300.lizard_attn import LIZARD_ERR_INVALID_ARG

    wl = WORKLOADS["decode"].replace(B=3, H=4, L=20)
    init = decode_initial_state(wl)
    st = _gpu_state_from(init, wl)
    st.pos[1] = -5
    inp = decode_step_inputs(wl, 0)
    y = gpu_decode_step(inp, init["mu"], wl.alpha, st).cpu()
    with pytest.raises(LizardError) as e:
        lizard_check_device_status()
    assert e.value.status == LIZARD_ERR_INVALID_ARG
    lizard_check_device_status()  # the error word was cleared
    seq = [0, 2]
    ost = dict(S=init["S"][seq].double().contiguous(), ring_k=init["ring_k"][seq].contiguous(),
               ring_v=init["ring_v"][seq].contiguous(), pos=init["pos"][seq].clone())
    sub = {n: inp[n][seq].contiguous() for n in ("q", "k", "v", "g")}
    y_ref = O.decode_step(sub["q"], sub["k"], sub["v"], sub["g"], init["mu"], wl.alpha, ost)
    assert rel_l2(y[seq], y_ref) <= 1e-2
    pos = st.pos.cpu()
    assert int(pos[0]) == wl.L + 1 and int(pos[2]) == wl.L + 1


def test_long_context_prefill_then_decode_all_heads():
    """B1 H32 L65536 d128 bf16, g ~ N(4,1), w64 m4: prefill of L tokens
    (one launch, sequence segments), its state handed to 128 decode steps.
    The oracle runs the recurrence over all L + 128 tokens for every head;
    the prefill rows and the decode steps must both match it (rel L2 <= 1e-2)."""
    wl = WORKLOADS["long_context"]
    n = wl.decode_steps
    inp = prefill_inputs(wl, L=wl.L + n)
    head = {k: (v[:, :, :wl.L].contiguous() if isinstance(v, torch.Tensor) and k != "mu" else v)
            for k, v in inp.items()}
    y_pre, st = gpu_prefill(head, wl.w)
    ys = []
    for t in range(wl.L, wl.L + n):
        step = {k: inp[k][:, :, t].contiguous() for k in ("q", "k", "v", "g")}
        ys.append(gpu_decode_step(step, inp["mu"], inp["alpha"], st).cpu())
    y_dec = torch.stack(ys, dim=2)  # [B, H, n, d]
    y_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], wl.w)
    err_pre = rel_l2(y_pre, y_ref[:, :, :wl.L])
    assert err_pre <= 1e-2, f"prefill rows: rel L2 {err_pre:.3e}"
    err_dec = rel_l2(y_dec, y_ref[:, :, wl.L:])
    assert err_dec <= 1e-2, f"decode rows: rel L2 {err_dec:.3e}"
    assert int(st.pos.cpu()[0]) == wl.L + n


_TIMEOUT_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from hybrid_gated_linear_attn_b300 import (LizardError, LizardState, lizard_attn_decode_step,
                                           lizard_check_device_status, lizard_state_init)
from hybrid_gated_linear_attn_b300 import lizard_attn as LA
B, H, d, w = 2, 4, 128, 64
st = LizardState(B, H, d, d, w, dtype=torch.bfloat16)
lizard_state_init(st)
x = torch.randn(B, H, d, dtype=torch.bfloat16, device="cuda")
mu = torch.randn(H, 4, d, dtype=torch.bfloat16, device="cuda")
lizard_attn_decode_step(x, x, x, x, mu, 1.0, st)
try:
    lizard_check_device_status()
    print("NO_TIMEOUT")
except LizardError as e:
    print("STATUS", e.status)
print("POS", st.pos.cpu().tolist())
lizard_check_device_status()  # cleared
print("SUM", float(torch.ones(1000, device="cuda").sum()))  # the context is still usable
"""


def test_forced_decode_timeout_is_reported_and_context_stays_usable(tmp_path):
    """Failure detection without a GPU fault: with the first wait capped at 0
    polls every decode CTA gives up at once, records the timeout, still
    waits (normal limit) for its copies, and retires; the host reads
    LIZARD_ERR_TIMEOUT and the process keeps using the GPU."""
    import os
    import subprocess
    import sys
    from hybrid_gated_linear_attn_b300 import lizard_attn as LA
    from hybrid_gated_linear_attn_b300 import lizard_attn_decode_step, lizard_check_device_status
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, LIZARD_DEBUG_DECODE_FIRST_WAIT_POLLS="0")
    out = subprocess.run([sys.executable, "-c", _TIMEOUT_CHILD, root], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert f"STATUS {LA.LIZARD_ERR_TIMEOUT}" in out.stdout, out.stdout
    assert "POS [1, 1]" in out.stdout, out.stdout  # the position still advances: every CTA counted itself
    assert "SUM 1000.0" in out.stdout, out.stdout
    # this process (no variable) decodes normally
    st = LizardState(1, 2, 128, 128, 64, dtype=torch.bfloat16)
    lizard_state_init(st)
    x = torch.randn(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    lizard_attn_decode_step(x, x, x, x, None, 1.0, st)
    lizard_check_device_status()
