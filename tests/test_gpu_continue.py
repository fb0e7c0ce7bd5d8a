"""Continued prefill (lizard_attn_prefill_continue) against the fp64 oracle.

A prompt of L1 tokens followed by a continuation of L2 tokens must give the
y and the state of one pass over all L1 + L2 tokens: the gate state carries
on (Lizard, gist.science/de section 2 item 1) and the first w - 1 new tokens
see the earlier ones in their anchor window (item 2).  The oracle runs the
whole sequence in one pass; y is compared element by element (relative L2,
<= 1e-4 fp32 / <= 1e-2 bf16), the final S likewise, ring and pos exactly.
"""
import zlib

import pytest
import torch

from hybrid_gated_linear_attn_b300 import (LizardError, LizardState, lizard_attn_decode_step,
                                           lizard_attn_prefill, lizard_attn_prefill_continue,
                                           lizard_check_device_status, lizard_state_init)
from hybrid_gated_linear_attn_b300 import lizard_attn as LA
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs, rel_l2
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs(name, dt, Bn, H, L, d, w, m, gm=3.0, gs=1.0, alpha=1.0):
    wl = WORKLOADS["llama3_8b"].replace(B=Bn, H=H, L=L, dk=d, dv=d, w=w, m=m, g_mean=gm, g_std=gs,
                                       alpha=alpha, dtype=dt, seed=zlib.crc32(name.encode()) % 1000)
    return prefill_inputs(wl)


def _dev(inp, lo, hi):
    return [inp[n][:, :, lo:hi].contiguous().cuda() for n in ("q", "k", "v", "g")]


def _check_state(st, inp, Ltot, S_ref, tol):
    errS = rel_l2(st.S.cpu(), S_ref)
    assert errS <= tol, f"final state rel L2 {errS:.3e}"
    assert torch.all(st.pos.cpu() == Ltot)
    w = st.w
    for p in range(max(0, Ltot - w), Ltot):
        assert torch.equal(st.ring_k[:, :, p % w].cpu(), inp["k"][:, :, p]), p
        assert torch.equal(st.ring_v[:, :, p % w].cpu(), inp["v"][:, :, p]), p


def _run_pieces(inp, w, pieces, first_is_prefill=True):
    """Feed the sequence in pieces: a prefill, then continuations."""
    Bn, H, _, d = inp["q"].shape
    mu = inp["mu"].cuda()
    st = LizardState(Bn, H, d, d, w, dtype=inp["q"].dtype)
    ys, lo = [], 0
    for i, n in enumerate(pieces):
        q, k, v, g = _dev(inp, lo, lo + n)
        if i == 0 and first_is_prefill:
            ys.append(lizard_attn_prefill(q, k, v, g, mu, inp["alpha"], w, state=st))
        else:
            if i == 0:
                lizard_state_init(st)
            ys.append(lizard_attn_prefill_continue(q, k, v, g, mu, inp["alpha"], st))
        lo += n
    torch.cuda.synchronize()
    lizard_check_device_status()
    return torch.cat([y.cpu() for y in ys], dim=2), st


CASES = [
    # name, dtype, B, H, pieces, d, w, m, g_mean, g_std, alpha
    # warp-specialised tensor-core path (bf16, d = 128 or 64, w <= 65)
    ("ws_two_pieces", "bf16", 2, 2, (200, 150), 128, 64, 4, 3.0, 1.0, 1.0),
    ("ws_short_history", "bf16", 1, 3, (10, 130), 128, 64, 4, 3.0, 1.0, 1.0),
    ("ws_short_continuation", "bf16", 1, 2, (300, 20), 128, 64, 4, 3.0, 1.0, 0.7),
    ("ws_chunk_aligned", "bf16", 2, 2, (128, 64, 192), 128, 64, 4, 3.0, 1.0, 1.0),
    ("ws_window_33", "bf16", 1, 2, (77, 150, 3), 128, 33, 2, 3.0, 1.0, 1.0),
    ("ws_window_one", "bf16", 1, 2, (100, 90), 128, 1, 3, 3.0, 1.0, 1.0),
    ("ws_window_65", "bf16", 1, 2, (70, 140), 128, 65, 4, 3.0, 1.0, 1.0),
    ("ws_strong_decay", "bf16", 1, 2, (300, 260), 128, 64, 4, -8.0, 4.0, 1.0),
    ("ws_segments", "bf16", 1, 2, (500, 3000), 128, 64, 4, 3.0, 1.0, 1.0),
    ("ws_segments_short_history", "bf16", 1, 1, (5, 2100), 128, 48, 4, 0.0, 2.0, 0.5),
    ("ws_segments_window_one", "bf16", 1, 2, (300, 1500), 128, 1, 2, 3.0, 1.0, 1.0),
    ("ws_d64_two_pieces", "bf16", 2, 2, (200, 150), 64, 64, 4, 3.0, 1.0, 1.0),
    ("ws_d64_short_history", "bf16", 1, 3, (10, 130, 70), 64, 48, 4, 3.0, 1.0, 1.0),
    ("ws_d64_strong_decay", "bf16", 1, 2, (300, 260), 64, 64, 4, -8.0, 4.0, 1.0),
    ("ws_d64_window_65", "bf16", 1, 2, (70, 140), 64, 65, 4, 3.0, 1.0, 1.0),
    # tensor-core path with a two-chunk window band (bf16, d = 128, w > 65)
    ("tc_window_100", "bf16", 1, 2, (300, 200), 128, 100, 4, 3.0, 1.0, 1.0),
    ("tc_window_128_short_history", "bf16", 1, 2, (30, 200, 70), 128, 128, 16, 3.0, 1.0, 1.0),
    ("tc_strong_decay", "bf16", 1, 2, (129, 300), 128, 80, 4, -8.0, 4.0, 0.5),
    # CUDA-core path (fp32, or bf16 d = 64 with w > 65)
    ("simt_f32_d128", "f32", 1, 2, (150, 130), 128, 64, 4, 3.0, 1.0, 1.0),
    ("simt_f32_d64", "f32", 2, 2, (37, 100, 64), 64, 16, 4, 3.0, 1.0, 0.5),
    ("ws_d64_w100", "bf16", 1, 2, (90, 160), 64, 100, 4, 3.0, 1.0, 1.0),
    ("simt_f32_window_one", "f32", 1, 2, (50, 60), 64, 1, 2, 3.0, 1.0, 0.7),
    # head dim 256 (CUDA cores, value slices; the ring hand-off after the slices)
    ("simt_bf16_d256", "bf16", 1, 2, (70, 90, 5), 256, 64, 4, 3.0, 1.0, 1.0),
    ("simt_f32_d256_short_history", "f32", 2, 1, (10, 100), 256, 100, 16, 0.0, 2.0, 0.5),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pieces_match_one_pass(case):
    name, dt, Bn, H, pieces, d, w, m, gm, gs, alpha = case
    Ltot = sum(pieces)
    inp = _inputs(name, dt, Bn, H, Ltot, d, w, m, gm, gs, alpha)
    y_gpu, st = _run_pieces(inp, w, pieces)
    y_ref, S_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], alpha, w, state=True)
    tol = TOL[inp["q"].dtype]
    err = rel_l2(y_gpu, y_ref)
    assert err <= tol, f"rel L2 {err:.3e} > {tol}"
    assert torch.isfinite(y_gpu.float()).all()
    _check_state(st, inp, Ltot, S_ref, tol)


@pytest.mark.parametrize("dt,d,w", [("bf16", 128, 64), ("bf16", 128, 100), ("bf16", 64, 64), ("f32", 64, 16)])
def test_continue_from_empty_state_is_a_prefill(dt, d, w):
    inp = _inputs(f"empty_{dt}_{d}_{w}", dt, 2, 2, 230, d, w, 4)
    y_gpu, st = _run_pieces(inp, w, (230,), first_is_prefill=False)
    y_pre, st_pre = _run_pieces(inp, w, (230,))
    tol = TOL[inp["q"].dtype]
    assert rel_l2(y_gpu, y_pre.double()) <= tol
    assert torch.equal(st.pos.cpu(), st_pre.pos.cpu())
    assert torch.equal(st.ring_k.cpu(), st_pre.ring_k.cpu())
    assert rel_l2(st.S.cpu(), st_pre.S.cpu().double()) <= tol


def test_empty_continuation_leaves_the_state():
    inp = _inputs("empty_cont", "bf16", 1, 2, 100, 128, 64, 4)
    _, st = _run_pieces(inp, 64, (100,))
    S, rk, pos = st.S.clone(), st.ring_k.clone(), st.pos.clone()
    e = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device="cuda")
    y = lizard_attn_prefill_continue(e, e, e, e, inp["mu"].cuda(), 1.0, st)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(S, st.S) and torch.equal(rk, st.ring_k) and torch.equal(pos, st.pos)


@pytest.mark.parametrize("dt,d,w", [("bf16", 128, 64), ("bf16", 128, 128), ("bf16", 64, 64), ("f32", 128, 40)])
def test_sequences_at_different_positions(dt, d, w):
    """One call continues sequences that have consumed 0, 5 and 300 tokens:
    the state is written by hand from the oracle (S, ring slots p % w, pos)."""
    p0s, L2, H = [0, 5, 300], 150, 2
    Lmax = max(p0s) + L2
    inp = _inputs(f"mixed_{dt}_{w}", dt, len(p0s), H, Lmax, d, w, 4)
    st = LizardState(len(p0s), H, d, d, w, dtype=inp["q"].dtype)
    lizard_state_init(st)
    torch.cuda.synchronize()
    q2, k2, v2, g2 = ([], [], [], [])
    refs = []
    for b, p0 in enumerate(p0s):
        sl = {n: inp[n][b:b + 1] for n in ("q", "k", "v", "g")}
        y_ref, S_b = O.forward(*(sl[n][:, :, :p0 + L2] for n in ("q", "k", "v", "g")), inp["mu"], inp["alpha"],
                               w, state=True)
        refs.append(y_ref[0, :, p0:])
        if p0 > 0:
            _, S_p = O.forward(*(sl[n][:, :, :p0] for n in ("q", "k", "v", "g")), inp["mu"], inp["alpha"], w,
                               state=True)
            st.S[b] = S_p[0].float().cuda()
            for p in range(max(0, p0 - w), p0):
                st.ring_k[b, :, p % w] = inp["k"][b, :, p].cuda()
                st.ring_v[b, :, p % w] = inp["v"][b, :, p].cuda()
        st.pos[b] = p0
        for lst, n in zip((q2, k2, v2, g2), ("q", "k", "v", "g")):
            lst.append(inp[n][b, :, p0:p0 + L2])
    q2, k2, v2, g2 = (torch.stack(t).contiguous().cuda() for t in (q2, k2, v2, g2))
    y = lizard_attn_prefill_continue(q2, k2, v2, g2, inp["mu"].cuda(), inp["alpha"], st)
    torch.cuda.synchronize()
    lizard_check_device_status()
    err = rel_l2(y.cpu(), torch.stack(refs))
    assert err <= TOL[inp["q"].dtype], f"rel L2 {err:.3e}"
    assert st.pos.cpu().tolist() == [p0 + L2 for p0 in p0s]


def test_decode_after_continuation():
    """prefill 90 + continue 100, then 3 decode steps, against the oracle's
    one pass over all 193 tokens."""
    w, steps = 64, 3
    inp = _inputs("decode_after", "bf16", 2, 2, 190 + steps, 128, w, 4)
    y_pre, st = _run_pieces(inp, w, (90, 100))
    mu = inp["mu"].cuda()
    ys = [y_pre]
    for t in range(190, 190 + steps):
        q, k, v, g = (inp[n][:, :, t].contiguous().cuda() for n in ("q", "k", "v", "g"))
        ys.append(lizard_attn_decode_step(q, k, v, g, mu, inp["alpha"], st).cpu()[:, :, None])
    torch.cuda.synchronize()
    y_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], inp["alpha"], w)
    err = rel_l2(torch.cat(ys, dim=2), y_ref)
    assert err <= TOL[torch.bfloat16], f"rel L2 {err:.3e}"


def test_bad_position_is_reported_and_stays_in_bounds():
    inp = _inputs("bad_pos", "bf16", 2, 2, 100, 128, 64, 4)
    _, st = _run_pieces(inp, 64, (100,))
    st.pos[1] = -5
    q, k, v, g = _dev(inp, 0, 70)
    lizard_attn_prefill_continue(q, k, v, g, inp["mu"].cuda(), 1.0, st)
    with pytest.raises(LizardError) as e:
        lizard_check_device_status()
    assert e.value.status == LA.LIZARD_ERR_INVALID_ARG
    lizard_check_device_status()  # cleared
    assert st.pos[0].item() == 170  # the other sequence's state is undefined now


def test_llama3_8b_chunked_prefill_all_units():
    """B4 H32 L4096 d128 bf16 fed as 2048 + 2048 tokens (the second a
    continuation) against one oracle pass over all 128 units; the final
    state's pos and ring exactly."""
    wl = WORKLOADS["llama3_8b"]
    inp = prefill_inputs(wl)
    y_gpu, st = _run_pieces(inp, wl.w, (2048, 2048))
    y_ref = O.forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["mu"], wl.alpha, wl.w)
    err = rel_l2(y_gpu, y_ref)
    assert err <= TOL[torch.bfloat16], f"rel L2 {err:.3e}"
    assert torch.all(st.pos.cpu() == wl.L)
    for p in range(wl.L - wl.w, wl.L):
        assert torch.equal(st.ring_k[:, :, p % wl.w].cpu(), inp["k"][:, :, p])
