"""Variants (lizard_variant): per-head anchor weights and grouped key/value
heads, through prefill, continued prefill, decode and the backward, on every
kernel path, against the fp64 oracle.

The oracle runs the plain operator per head with that head's alpha, on the
key/value heads expanded to every query head of their group (that is what
sharing means); the backward's dk, dv of a key/value head are the sums of
the oracle's per-query-head gradients over the group (the chain rule through
the sharing), d alpha_h the oracle's d alpha of head h.
"""
import zlib

import pytest
import torch

from hybrid_gated_linear_attn_b300 import (LizardState, lizard_attn_backward, lizard_attn_decode_step,
                                           lizard_attn_prefill, lizard_attn_prefill_continue,
                                           lizard_check_device_status)
from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs, rel_l2
from oracle import oracle as O
from tests.gpu_helpers import TOL, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs(name, dt, Bn, H, Hkv, L, d, w, m, gm=3.0, gs=1.0):
    seed = zlib.crc32(name.encode()) % 1000
    wl = WORKLOADS["llama3_8b"].replace(B=Bn, H=H, L=L, dk=d, dv=d, w=w, m=m, g_mean=gm, g_std=gs, dtype=dt, seed=seed)
    inp = prefill_inputs(wl)
    grp = H // Hkv
    inp["k"] = inp["k"][:, ::grp].contiguous()  # one key/value head per group
    inp["v"] = inp["v"][:, ::grp].contiguous()
    gen = torch.Generator().manual_seed(seed + 3)
    inp["alpha_h"] = (torch.rand(H, generator=gen) * 1.5 + 0.25).float()
    inp["dy"] = torch.randn(Bn, H, L, d, generator=gen).to(inp["q"].dtype)
    inp["group"] = grp
    return inp


def _expand(t, grp):
    return t.repeat_interleave(grp, dim=1)


def _oracle_y(inp, w, lo=0, hi=None):
    """y of every head over tokens [0, hi), rows lo.. returned."""
    grp, H = inp["group"], inp["q"].shape[1]
    hi = inp["q"].shape[2] if hi is None else hi
    k, v = _expand(inp["k"], grp), _expand(inp["v"], grp)
    ys = []
    for h in range(H):
        sl = lambda t: t[:, h:h + 1, :hi]  # noqa: E731
        ys.append(O.forward(sl(inp["q"]), sl(k), sl(v), sl(inp["g"]), inp["mu"][h:h + 1],
                            float(inp["alpha_h"][h]), w)[:, 0, lo:])
    return torch.stack(ys, dim=1)


def _dev(inp, *names):
    return [inp[n].cuda() for n in names]


CASES = [
    # name, dtype, B, H, Hkv, L, d, w, m
    ("ws_gqa2", "bf16", 2, 4, 2, 200, 128, 64, 4),
    ("ws_mqa", "bf16", 1, 4, 1, 150, 128, 48, 2),
    ("ws_segments_gqa", "bf16", 1, 4, 2, 1600, 128, 64, 4),
    ("tc_gqa2", "bf16", 1, 4, 2, 260, 128, 100, 4),
    ("simt_f32_gqa2", "f32", 1, 4, 2, 150, 64, 16, 4),
    ("ws_d64_mqa", "bf16", 2, 2, 1, 130, 64, 32, 3),
    ("ws_d64_gqa2", "bf16", 2, 4, 2, 200, 64, 64, 4),
    ("ws_d64_w100_gqa2", "bf16", 1, 4, 2, 160, 64, 100, 4),
    ("ws_per_head_alpha_only", "bf16", 1, 3, 3, 140, 128, 64, 4),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_variants(case):
    name, dt, Bn, H, Hkv, L, d, w, m = case
    inp = _inputs(name, dt, Bn, H, Hkv, L, d, w, m)
    q, k, v, g, mu, ah = _dev(inp, "q", "k", "v", "g", "mu", "alpha_h")
    st = LizardState(Bn, H, d, d, w, dtype=q.dtype)
    y = lizard_attn_prefill(q, k, v, g, mu, 1.0, w, state=st, alpha_h=ah, Hkv=Hkv)
    torch.cuda.synchronize()
    lizard_check_device_status()
    err = rel_l2(y.cpu(), _oracle_y(inp, w))
    assert err <= TOL[q.dtype], f"rel L2 {err:.3e}"
    # the ring keeps each query head's window: its group's key/value head
    kx = _expand(inp["k"], inp["group"])
    for p in range(max(0, L - w), L):
        assert torch.equal(st.ring_k[:, :, p % w].cpu(), kx[:, :, p])


@pytest.mark.parametrize("dt,d,w", [("bf16", 128, 64), ("bf16", 128, 100), ("bf16", 64, 64), ("f32", 64, 16)])
def test_continue_and_decode_variants(dt, d, w):
    """prefill 90 + continue 60 + 3 decode steps, grouped heads, per-head alpha."""
    Bn, H, Hkv, steps = 2, 4, 2, 3
    L = 150 + steps
    inp = _inputs(f"cd_{dt}_{d}_{w}", dt, Bn, H, Hkv, L, d, w, 4)
    q, k, v, g, mu, ah = _dev(inp, "q", "k", "v", "g", "mu", "alpha_h")
    st = LizardState(Bn, H, d, d, w, dtype=q.dtype)
    ys = [lizard_attn_prefill(q[:, :, :90].contiguous(), k[:, :, :90].contiguous(), v[:, :, :90].contiguous(),
                              g[:, :, :90].contiguous(), mu, 1.0, w, state=st, alpha_h=ah, Hkv=Hkv)]
    ys.append(lizard_attn_prefill_continue(*(t[:, :, 90:150].contiguous() for t in (q, k, v, g)), mu, 1.0, st,
                                           alpha_h=ah, Hkv=Hkv))
    for t in range(150, L):
        ys.append(lizard_attn_decode_step(*(x[:, :, t].contiguous() for x in (q, k, v, g)), mu, 1.0, st,
                                          alpha_h=ah, Hkv=Hkv)[:, :, None])
    torch.cuda.synchronize()
    lizard_check_device_status()
    err = rel_l2(torch.cat([y.cpu() for y in ys], dim=2), _oracle_y(inp, w))
    assert err <= TOL[q.dtype], f"rel L2 {err:.3e}"


BWD_CASES = [
    # name, dtype, B, H, Hkv, L, d, w, m
    ("bwd_tc_gqa2", "bf16", 1, 4, 2, 200, 128, 64, 4),
    ("bwd_tc_d64_gqa2", "bf16", 1, 4, 2, 200, 64, 64, 4),
    ("bwd_tc_mqa", "bf16", 2, 2, 1, 130, 128, 33, 2),
    ("bwd_simt_f32_gqa2", "f32", 1, 4, 2, 120, 64, 16, 4),
    ("bwd_simt_bf16_w100", "bf16", 1, 4, 2, 150, 128, 100, 4),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_backward_variants(case):
    name, dt, Bn, H, Hkv, L, d, w, m = case
    inp = _inputs(name, dt, Bn, H, Hkv, L, d, w, m)
    grp = inp["group"]
    q, k, v, g, mu, ah, dy = _dev(inp, "q", "k", "v", "g", "mu", "alpha_h", "dy")
    dq, dk, dv, dg, dmu, dal = (None if t is None else t.cpu() for t in
                                lizard_attn_backward(q, k, v, g, mu, 1.0, w, dy, alpha_h=ah, Hkv=Hkv))
    torch.cuda.synchronize()
    lizard_check_device_status()
    kx, vx = _expand(inp["k"], grp), _expand(inp["v"], grp)
    refs = []
    for h in range(H):
        sl = lambda t: t[:, h:h + 1]  # noqa: E731
        refs.append(O.backward(sl(inp["q"]), sl(kx), sl(vx), sl(inp["g"]), inp["mu"][h:h + 1],
                               float(inp["alpha_h"][h]), w, sl(inp["dy"]).double()))
    cat = lambda n: torch.cat([r[n] for r in refs], dim=1)  # noqa: E731
    dk_ref = cat("dk").reshape(Bn, H // grp, grp, L, d).sum(2)
    dv_ref = cat("dv").reshape(Bn, H // grp, grp, L, d).sum(2)
    tol = TOL[q.dtype]
    errs = {"dq": rel_l2(dq, cat("dq")), "dk": rel_l2(dk, dk_ref), "dv": rel_l2(dv, dv_ref),
            "dg": rel_l2(dg, cat("dg")), "dmu": rel_l2(dmu, torch.cat([r["dmu"] for r in refs], dim=0))}
    # d alpha_h = sum_t dy_t . ya_t over head h: a sum of terms of both
    # signs, bounded by tol * sum |dy ya| of that head
    for h in range(H):
        _, _, ya = O.forward(kx[:, h:h + 1] * 0 + inp["q"][:, h:h + 1], kx[:, h:h + 1], vx[:, h:h + 1],
                             inp["g"][:, h:h + 1], inp["mu"][h:h + 1], float(inp["alpha_h"][h]), w, branches=True)
        scale = float((inp["dy"][:, h:h + 1].double() * ya).abs().sum())
        errs[f"dalpha[{h}]"] = abs(float(dal[h]) - float(refs[h]["dalpha"])) / max(scale, 1e-30)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"above {tol}: {bad} (all: {errs})"
