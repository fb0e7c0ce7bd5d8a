"""ctypes front end of the fp64 CPU oracle (``lizard_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test-suite, the smoke check and the benchmark's
CPU-baseline leg use this module.  The library under ``hybrid_gated_linear_attn_b300``
never imports it, and it never imports that library (the seeded input
generators are the one module both sides read).

Tensors are CPU torch tensors; bf16 inputs are passed as their raw 16-bit
patterns and widened to fp64 inside the C code, so the oracle sees exactly
the bits the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lizard_oracle.c")
LIB = os.path.join(HERE, "liblizard_oracle.so")

_F32, _BF16 = 0, 1
_lock = threading.Lock()
_libs: dict = {}


def build(out: str = LIB, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with gcc (optionally with one planted mistake)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-shared", "-fPIC", "-pthread",
           SRC, "-o", tmp, "-lm"]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str = LIB) -> ctypes.CDLL:
    with _lock:
        if path in _libs:
            return _libs[path]
        if path == LIB:
            build()
        lib = ctypes.CDLL(path)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_forward.argtypes = [I, P, P, P, P, P, D, I, I, I, I, I, I, I, I,
                                       P, P, P, I, P, P, P, P, I]
        lib.oracle_forward.restype = I
        lib.oracle_decode_step.argtypes = [I, P, P, P, P, P, D, I, I, I, I, I, I, P, P, P, P, P]
        lib.oracle_decode_step.restype = I
        lib.oracle_gla_product_form.argtypes = [I, P, P, P, P, I, I, I, P, P]
        lib.oracle_gla_product_form.restype = I
        lib.oracle_backward.argtypes = [I, P, P, P, P, P, D, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, I]
        lib.oracle_backward.restype = I
        lib.oracle_log_sigmoid.argtypes = [D]
        lib.oracle_log_sigmoid.restype = D
        _libs[path] = lib
        return lib


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return _F32
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"oracle takes fp32 or bf16 inputs, got {t.dtype}")


def _c(t):
    """Contiguous CPU tensor (or None) and its address."""
    if t is None:
        return None, None
    t = t.detach().to("cpu").contiguous()
    return t, ctypes.c_void_p(t.data_ptr())


def default_threads() -> int:
    return os.cpu_count() or 1


def forward(q, k, v, g, mu, alpha, w, *, S0=None, hist_k=None, hist_v=None,
            branches=False, state=False, threads=None, lib=None):
    """Run the operator on [B,H,L,d] inputs (or [U,L,d] units, H from mu).

    S0 [B,H,dk,dv] (fp64 or fp32) is the initial state, hist_k/hist_v
    [B,H,hlen,d] the tokens that precede the sequence (window history).
    Returns y (fp64) and, on request, the branches (yg, ya) and final S.
    """
    lib = lib or load()
    dt = _code(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    H, m = mu.shape[0], mu.shape[1]
    U = 1
    for s in lead:
        U *= s
    tensors = []

    def keep(t):
        t, p = _c(t)
        tensors.append(t)
        return p

    pq, pk, pv, pg = keep(q.to(q.dtype)), keep(k), keep(v), keep(g)
    pmu = keep(mu) if m > 0 else None
    pS0 = keep(S0.double()) if S0 is not None else None
    hlen = 0 if hist_k is None else hist_k.shape[-2]
    phk = keep(hist_k) if hlen else None
    phv = keep(hist_v) if hlen else None
    y = torch.empty(*lead, L, dv, dtype=torch.float64)
    yg = torch.empty_like(y) if branches else None
    ya = torch.empty_like(y) if branches else None
    S = torch.empty(*lead, dk, dv, dtype=torch.float64) if state else None
    rc = lib.oracle_forward(dt, pq, pk, pv, pg, pmu, float(alpha), U, 0, H, L, dk, dv, int(w), m,
                            pS0, phk, phv, hlen,
                            ctypes.c_void_p(y.data_ptr()),
                            ctypes.c_void_p(yg.data_ptr()) if branches else None,
                            ctypes.c_void_p(ya.data_ptr()) if branches else None,
                            ctypes.c_void_p(S.data_ptr()) if state else None,
                            threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    out = [y]
    if branches:
        out += [yg, ya]
    if state:
        out.append(S)
    return out[0] if len(out) == 1 else tuple(out)


def forward_units(q, k, v, g, mu, alpha, w, units, *, threads=None, lib=None, S0=None):
    """The operator on selected (b, h) units only: y[len(units), L, dv] fp64.

    ``units`` is a list of (b, h) pairs; inputs are [B,H,L,d].  Each unit
    runs the full recurrence over its own sequence.
    """
    lib = lib or load()
    ys = []
    for (b, h) in units:
        mu_h = mu[h:h + 1]
        s0 = None if S0 is None else S0[b, h][None]
        ys.append(forward(q[b, h][None], k[b, h][None], v[b, h][None], g[b, h][None],
                          mu_h, alpha, w, S0=s0, threads=1, lib=lib)[0])
    return torch.stack(ys)


def forward_units_parallel(q, k, v, g, mu, alpha, w, units, *, lib=None):
    """forward_units with one unit per thread (the C code releases the GIL)."""
    lib = lib or load()
    out = [None] * len(units)

    def run(i, bh):
        out[i] = forward_units(q, k, v, g, mu, alpha, w, [bh], lib=lib)[0]

    ths = [threading.Thread(target=run, args=(i, bh)) for i, bh in enumerate(units)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    return torch.stack(out)


def decode_step(q, k, v, g, mu, alpha, st: dict, *, lib=None):
    """One decode step on the oracle's own state dict (updated in place).

    st: S [B,H,dk,dv] fp64, ring_k/ring_v [B,H,w,d] (input dtype), pos [B] int64.
    Inputs q,k,g [B,H,dk], v [B,H,dv].  Returns y [B,H,dv] fp64.
    """
    lib = lib or load()
    dt = _code(q)
    B, H, dk = q.shape
    dv = v.shape[-1]
    w = st["ring_k"].shape[2]
    m = mu.shape[1]
    for key in ("S", "ring_k", "ring_v", "pos"):
        assert st[key].is_contiguous()
    assert st["S"].dtype == torch.float64 and st["pos"].dtype == torch.int64
    q, k, v, g = (t.contiguous() for t in (q, k, v, g))
    mu = mu.contiguous()
    y = torch.empty(B, H, dv, dtype=torch.float64)
    rc = lib.oracle_decode_step(dt, q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                                mu.data_ptr() if m > 0 else None, float(alpha), B, H, dk, dv, w, m,
                                st["S"].data_ptr(), st["ring_k"].data_ptr(), st["ring_v"].data_ptr(),
                                st["pos"].data_ptr(), y.data_ptr())
    if rc != 0:
        raise ValueError("oracle_decode_step rejected its arguments")
    return y


def backward(q, k, v, g, mu, alpha, w, dy, *, threads=None, lib=None) -> dict:
    """Gradients of sum(dy * y) for [B,H,L,d] inputs (or [U,L,d] units, H
    from mu) that start from the empty state.

    Returns fp64 tensors: dq, dk, dv, dg shaped like the inputs, dmu [H,m,dk]
    (summed over the batch) and dalpha (a 0-d tensor, summed over all units).
    """
    lib = lib or load()
    dt = _code(q)
    lead = q.shape[:-2]
    L, dk = q.shape[-2], q.shape[-1]
    dv = v.shape[-1]
    H, m = mu.shape[0], mu.shape[1]
    U = 1
    for s_ in lead:
        U *= s_
    tensors = []

    def keep(t):
        t, p = _c(t)
        tensors.append(t)
        return p

    pq, pk, pv, pg = keep(q), keep(k), keep(v), keep(g)
    pmu = keep(mu) if m > 0 else None
    pdy = keep(dy.double())
    dq = torch.empty(*lead, L, dk, dtype=torch.float64)
    dk_ = torch.empty_like(dq)
    dg = torch.empty_like(dq)
    dv_ = torch.empty(*lead, L, dv, dtype=torch.float64)
    dmu_u = torch.empty(U, m, dk, dtype=torch.float64)
    dalpha_u = torch.empty(U, dtype=torch.float64)
    rc = lib.oracle_backward(dt, pq, pk, pv, pg, pmu, float(alpha), U, 0, H, L, dk, dv, int(w), m, pdy,
                             ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk_.data_ptr()),
                             ctypes.c_void_p(dv_.data_ptr()), ctypes.c_void_p(dg.data_ptr()),
                             ctypes.c_void_p(dmu_u.data_ptr()), ctypes.c_void_p(dalpha_u.data_ptr()),
                             threads or default_threads())
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    # unit u = b * H + h: sum dmu over the batch for each head
    dmu = dmu_u.reshape(U // H if H else 0, H, m, dk).sum(0) if U else torch.zeros(H, m, dk, dtype=torch.float64)
    return {"dq": dq, "dk": dk_, "dv": dv_, "dg": dg, "dmu": dmu, "dalpha": dalpha_u.sum()}


def gla_product_form(q, k, v, g, S0=None, *, lib=None):
    """Gate branch of one unit ([L,d] inputs) by the O(L^3) product form."""
    lib = lib or load()
    L, dk = q.shape
    dv = v.shape[-1]
    q, k, v, g = (t.contiguous() for t in (q, k, v, g))
    s0 = None if S0 is None else S0.double().contiguous()
    yg = torch.empty(L, dv, dtype=torch.float64)
    rc = lib.oracle_gla_product_form(_code(q), q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                                     L, dk, dv, s0.data_ptr() if s0 is not None else None, yg.data_ptr())
    if rc != 0:
        raise ValueError("oracle_gla_product_form rejected its arguments")
    return yg


def log_sigmoid(x: float, *, lib=None) -> float:
    lib = lib or load()
    return lib.oracle_log_sigmoid(float(x))


def gate_projection(x, W, H):
    """Gate logits of the gated linear attention from the layer input: the
    gate module Gamma = sigmoid(W_gamma x) of Lizard (gist.science/de
    section 2 item 1) feeds the operator its logits g = W_gamma x.

    x [B, L, dmodel], W [H * dk, dmodel] (a linear layer's weight), both
    widened exactly to fp64; returns g [B, H, L, dk] fp64 (head-major, the
    operator's layout): g[b, h, t, i] = sum_c x[b, t, c] W[h dk + i, c].
    """
    B, L, dm = x.shape
    N = W.shape[0]
    dk = N // H
    g = x.double().reshape(B * L, dm) @ W.double().t()
    return g.reshape(B, L, H, dk).permute(0, 2, 1, 3).contiguous()
