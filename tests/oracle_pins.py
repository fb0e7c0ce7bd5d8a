"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each pin takes an oracle library handle and raises AssertionError when the
oracle disagrees with:
  * a library routine on a special case (scipy's log_expit, PyTorch's
    scaled_dot_product_attention, plain fp64 matmuls of causal linear
    attention),
  * a closed form (single token, constant gate, all gates open),
  * a structurally different formulation (the O(L^3) product form of the gate
    branch), or
  * an invariant of the definition (decode continues prefill, a prefill split
    in two equals the whole, linearity in v and alpha).

The pins are plain functions so that the mutation test can run all of them
against oracle builds with a planted mistake and require each mistake to be
caught by at least one pin.
"""
from __future__ import annotations

import math

import scipy.special
import torch
import torch.nn.functional as F

from oracle import oracle as O

f64 = torch.float64


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _qkvg(seed, B, H, L, dk, dv, g_mean=0.0, g_std=2.0, m=3, dtype=torch.float32):
    gen = _gen(seed)
    q = (torch.randn(B, H, L, dk, generator=gen) / math.sqrt(dk)).to(dtype)
    k = (torch.randn(B, H, L, dk, generator=gen) / math.sqrt(dk)).to(dtype)
    v = torch.randn(B, H, L, dv, generator=gen).to(dtype)
    g = (torch.randn(B, H, L, dk, generator=gen) * g_std + g_mean).to(dtype)
    mu = (torch.randn(H, m, dk, generator=gen) / 8).to(dtype)
    return q, k, v, g, mu


def _close(a, b, tol, what):
    a = a.double()
    b = b.double()
    err = float((a - b).abs().max())
    scale = float(b.abs().max()) + 1e-300
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} vs scale {scale:.3e} (tol {tol})"


# --- gate ------------------------------------------------------------------

def pin_log_sigmoid_vs_scipy(lib):
    xs = [-1e4, -745.0, -100.0, -30.0, -5.0, -1.0, -1e-3, 0.0, 1e-3, 1.0, 5.0, 30.0, 100.0, 745.0, 1e4]
    for x in xs:
        ref = float(scipy.special.log_expit(x))
        got = O.log_sigmoid(x, lib=lib)
        assert abs(got - ref) <= 1e-14 * max(1.0, abs(ref)) + 1e-300, f"log_sigmoid({x}): {got} vs {ref}"


# --- gate branch -----------------------------------------------------------

def pin_recurrence_equals_product_form(lib):
    for (L, dk, dv, seed) in [(11, 5, 7, 1), (9, 6, 6, 2), (1, 4, 3, 3)]:
        q, k, v, g, mu = _qkvg(seed, 1, 1, L, dk, dv, g_mean=0.5, g_std=2.0)
        S0 = torch.randn(1, 1, dk, dv, generator=_gen(seed + 100), dtype=f64)
        for s0 in (None, S0):
            y, yg, ya = O.forward(q, k, v, g, mu, 0.7, 4, S0=s0, branches=True, lib=lib)
            ref = O.gla_product_form(q[0, 0], k[0, 0], v[0, 0], g[0, 0],
                                     None if s0 is None else s0[0, 0], lib=lib)
            _close(yg[0, 0], ref, 1e-12, f"gate branch vs product form L={L} dk={dk} dv={dv}")
            # alpha = 0 leaves the gate branch alone in y
            y0 = O.forward(q, k, v, g, mu, 0.0, 4, S0=s0, lib=lib)
            _close(y0[0, 0], ref, 1e-12, "y(alpha=0) vs product form")


def pin_open_gates_are_causal_linear_attention(lib):
    # g = +inf gives sigmoid(g) = 1 exactly: no decay, so the gate branch is
    # causal linear attention  yg = tril(Q K^T) V + Q S0.
    B, H, L, dk, dv = 2, 2, 37, 8, 8
    q, k, v, g, mu = _qkvg(7, B, H, L, dk, dv)
    g = torch.full_like(g, float("inf"))
    S0 = torch.randn(B, H, dk, dv, generator=_gen(8), dtype=f64)
    _, yg, _ = O.forward(q, k, v, g, mu, 1.0, 5, S0=S0, branches=True, lib=lib)
    qd, kd, vd = q.double(), k.double(), v.double()
    A = torch.tril(qd @ kd.transpose(-1, -2))
    ref = A @ vd + qd @ S0
    _close(yg, ref, 1e-12, "open gates vs causal linear attention")


def pin_constant_gate_geometric_form(lib):
    # A gate that is constant over time, gamma_i per key dim, gives
    # yg_t = sum_{s<=t} sum_i q_ti k_si gamma_i^(t-s) v_s.
    L, dk, dv = 23, 6, 5
    q, k, v, g, mu = _qkvg(11, 1, 1, L, dk, dv)
    gi = torch.randn(dk, generator=_gen(12)) * 1.5
    g = gi.expand(1, 1, L, dk).contiguous()
    _, yg, _ = O.forward(q, k, v, g, mu, 1.0, 3, branches=True, lib=lib)
    gamma = torch.sigmoid(gi.double())
    t = torch.arange(L, dtype=f64)
    lag = t[:, None] - t[None, :]                          # t - s
    causal = lag >= 0
    decay = gamma[None, None, :] ** lag.clamp(min=0)[:, :, None]   # [t,s,i]
    A = torch.einsum("ti,si,tsi->ts", q[0, 0].double(), k[0, 0].double(), decay) * causal
    ref = A @ v[0, 0].double()
    _close(yg[0, 0], ref, 1e-12, "constant gate vs geometric closed form")


# --- anchor branch ---------------------------------------------------------

def pin_full_window_is_causal_softmax(lib):
    # w >= L and m = 0: the anchor branch is causal softmax attention with no
    # scale, i.e. scaled_dot_product_attention(is_causal=True, scale=1).
    B, H, L, d = 2, 3, 29, 8
    q, k, v, g, mu = _qkvg(21, B, H, L, d, d, m=0)
    q = q * 4  # sharper distributions
    for w in (L, L + 5):
        _, _, ya = O.forward(q, k, v, g, mu, 1.0, w, branches=True, lib=lib)
        ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double(), is_causal=True, scale=1.0)
        _close(ya, ref, 1e-12, f"full window (w={w}) vs causal SDPA")


def pin_window_and_sinks_vs_masked_sdpa(lib):
    # Sliding window of w keys (current token included) plus m sink keys of
    # value zero: SDPA over keys [mu ; K] and values [0 ; V] with a boolean
    # mask that admits every sink and keys t-w < s <= t.
    B, H, L, d, m = 1, 2, 33, 8, 3
    for w in (1, 2, 5, 16):
        q, k, v, g, mu = _qkvg(30 + w, B, H, L, d, d, m=m)
        q = q * 3
        _, _, ya = O.forward(q, k, v, g, mu, 1.0, w, branches=True, lib=lib)
        keys = torch.cat([mu.double()[None].expand(B, H, m, d), k.double()], dim=2)
        vals = torch.cat([torch.zeros(B, H, m, d, dtype=f64), v.double()], dim=2)
        t = torch.arange(L)[:, None]
        s = torch.arange(L)[None, :]
        band = (s <= t) & (s > t - w)
        mask = torch.cat([torch.ones(L, m, dtype=torch.bool), band], dim=1)
        ref = F.scaled_dot_product_attention(q.double(), keys, vals, attn_mask=mask, scale=1.0)
        _close(ya, ref, 1e-12, f"window w={w} with {m} sinks vs masked SDPA")


def pin_meta_logits_minus_inf_vanish(lib):
    # Sinks whose logits underflow (q > 0, mu << 0) weigh nothing: y equals
    # the m = 0 result.
    B, H, L, d = 1, 2, 19, 8
    q, k, v, g, mu = _qkvg(41, B, H, L, d, d, m=4)
    q = q.abs() + 0.05
    mu_neg = torch.full_like(mu, -1e3)
    y_sink = O.forward(q, k, v, g, mu_neg, 0.9, 6, lib=lib)
    y_none = O.forward(q, k, v, g, mu[:, :0], 0.9, 6, lib=lib)
    _close(y_sink, y_none, 1e-15, "vanishing sinks vs m=0")


def pin_single_token_closed_form(lib):
    # L = 1 from a zero state: yg = (q.k) v and the window holds only token 0:
    # y = (q.k) v + alpha e^{q.k} v / (e^{q.k} + sum_j e^{q.mu_j}).
    B, H, d, m = 1, 3, 6, 4
    q, k, v, g, mu = _qkvg(51, B, H, 1, d, d, m=m)
    alpha = 0.37
    for w in (1, 4):
        y = O.forward(q, k, v, g, mu, alpha, w, lib=lib)
        for h in range(H):
            qd, kd, vd = q[0, h, 0].double(), k[0, h, 0].double(), v[0, h, 0].double()
            a = float(qd @ kd)
            c = (mu[h].double() @ qd)
            Z = math.exp(a) + float(torch.exp(c).sum())
            ref = a * vd + alpha * math.exp(a) / Z * vd
            _close(y[0, h, 0], ref, 1e-13, f"single token closed form h={h}")


# --- combine and invariants -------------------------------------------------

def pin_linearity_in_alpha_and_v(lib):
    B, H, L, d = 1, 2, 21, 6
    q, k, v, g, mu = _qkvg(61, B, H, L, d, d, m=2)
    # quantise v, v2 to multiples of 1/256 so that v + v2 is exact in fp32
    v = (v * 256).round() / 256
    v2 = (torch.randn(v.shape, generator=_gen(62)) * 256).round() / 256
    y0 = O.forward(q, k, v, g, mu, 0.0, 5, lib=lib)
    y1 = O.forward(q, k, v, g, mu, 1.0, 5, lib=lib)
    ya = O.forward(q, k, v, g, mu, 2.5, 5, lib=lib)
    _close(ya, y0 + 2.5 * (y1 - y0), 1e-12, "linear in alpha")
    ys = O.forward(q, k, v + v2, g, mu, 0.8, 5, lib=lib)
    yv = O.forward(q, k, v, g, mu, 0.8, 5, lib=lib) + O.forward(q, k, v2, g, mu, 0.8, 5, lib=lib)
    _close(ys, yv, 1e-12, "linear in v")


def pin_split_prefill_equals_whole(lib):
    # Prefill of L1 tokens, then prefill of the rest from the returned state
    # and the last w-1 tokens as window history, equals one prefill of all.
    B, H, L, d, m = 1, 2, 40, 6, 2
    q, k, v, g, mu = _qkvg(71, B, H, L, d, d, m=m)
    for (L1, w) in [(17, 5), (3, 9), (20, 1)]:
        y_all = O.forward(q, k, v, g, mu, 0.6, w, lib=lib)
        _, S1 = O.forward(q[:, :, :L1], k[:, :, :L1], v[:, :, :L1], g[:, :, :L1], mu, 0.6, w,
                          state=True, lib=lib)
        hl = min(L1, w - 1)
        hk = k[:, :, L1 - hl:L1] if hl else None
        hv = v[:, :, L1 - hl:L1] if hl else None
        y2 = O.forward(q[:, :, L1:], k[:, :, L1:], v[:, :, L1:], g[:, :, L1:], mu, 0.6, w,
                       S0=S1, hist_k=hk, hist_v=hv, lib=lib)
        _close(y2, y_all[:, :, L1:], 1e-12, f"split prefill L1={L1} w={w}")


def pin_decode_continues_prefill(lib):
    # Prefill L tokens, load the ring with the last min(L, w) tokens, run n
    # decode steps: equals a prefill of L + n tokens, row by row.
    B, H, d, m, n = 2, 2, 6, 3, 7
    for (L, w) in [(13, 4), (3, 8), (10, 1)]:
        q, k, v, g, mu = _qkvg(80 + L, B, H, L + n, d, d, m=m)
        y_all = O.forward(q, k, v, g, mu, 0.8, w, lib=lib)
        _, S = O.forward(q[:, :, :L], k[:, :, :L], v[:, :, :L], g[:, :, :L], mu, 0.8, w, state=True, lib=lib)
        ring_k = torch.zeros(B, H, w, d)
        ring_v = torch.zeros(B, H, w, d)
        for p in range(max(0, L - w), L):
            ring_k[:, :, p % w] = k[:, :, p]
            ring_v[:, :, p % w] = v[:, :, p]
        st = dict(S=S.contiguous(), ring_k=ring_k, ring_v=ring_v, pos=torch.full((B,), L, dtype=torch.int64))
        for t in range(L, L + n):
            yt = O.decode_step(q[:, :, t], k[:, :, t], v[:, :, t], g[:, :, t], mu, 0.8, st, lib=lib)
            _close(yt, y_all[:, :, t], 1e-12, f"decode step t={t} (L={L}, w={w})")
        assert int(st["pos"][0]) == L + n


def pin_sink_free_weights_sum_to_one(lib):
    # With v = 1 and m = 0 the anchor branch is the sum of the window's
    # softmax weights: exactly 1 for every token.  With sinks it is below 1.
    B, H, L, d = 1, 2, 15, 5
    q, k, v, g, mu = _qkvg(91, B, H, L, d, d, m=3)
    ones = torch.ones_like(v)
    _, _, ya = O.forward(q, k, ones, g, mu[:, :0], 1.0, 4, branches=True, lib=lib)
    _close(ya, torch.ones_like(ya, dtype=f64), 1e-15, "sink-free weights sum to 1")
    _, _, ya = O.forward(q, k, ones, g, mu, 1.0, 4, branches=True, lib=lib)
    assert float(ya.max()) < 1.0


# --- backward ----------------------------------------------------------------

def _grid_inputs(seed, B, H, L, d, m):
    """fp32 inputs on a 2^-8 grid in [-2, 2] (g in [-3, 3]), so that x +- h
    stays exact in fp32 for the step sizes used below."""
    gen = _gen(seed)

    def grid(shape, scale):
        return (torch.round(torch.rand(*shape, generator=gen) * 2 * scale * 256 - scale * 256) / 256).float()

    return (grid((B, H, L, d), 1.0), grid((B, H, L, d), 1.0), grid((B, H, L, d), 2.0), grid((B, H, L, d), 3.0),
            grid((H, m, d), 1.0))


def _loss(q, k, v, g, mu, alpha, w, dy, lib):
    return float((O.forward(q, k, v, g, mu, alpha, w, lib=lib) * dy).sum())


def _fd_grad(x, f, h):
    """Central differences of f at every element of x (a CPU fp32 tensor),
    Richardson-extrapolated over steps h and h/2 (error O(h^4))."""
    out = torch.empty(x.shape, dtype=f64)
    flat = x.reshape(-1)
    for i in range(flat.numel()):
        x0 = float(flat[i])
        vals = []
        for step in (h, h / 2):
            flat[i] = x0 + step
            fp = f()
            flat[i] = x0 - step
            fm = f()
            vals.append((fp - fm) / (2 * step))
        flat[i] = x0
        out.reshape(-1)[i] = (4 * vals[1] - vals[0]) / 3
    return out


def pin_backward_vs_finite_differences(lib):
    # Gradients of sum(dy * y) against finite differences of the forward
    # oracle, element by element, for every input, mu and alpha.
    for (seed, L, d, w, m) in ((101, 9, 4, 3, 2), (102, 70, 3, 5, 1)):
        B, H, alpha = 1, 2, 0.7
        q, k, v, g, mu = _grid_inputs(seed, B, H, L, d, m)
        dy = torch.randn(B, H, L, d, generator=_gen(seed + 1), dtype=f64)
        got = O.backward(q, k, v, g, mu, alpha, w, dy, lib=lib)
        f = lambda: _loss(q, k, v, g, mu, alpha, w, dy, lib)  # noqa: E731
        h = 2.0 ** -7
        for name, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dmu", mu)):
            _close(got[name], _fd_grad(x, f, h), 1e-7, f"{name} vs finite differences (L={L})")
        da = [(_loss(q, k, v, g, mu, alpha + st, w, dy, lib) - _loss(q, k, v, g, mu, alpha - st, w, dy, lib))
              / (2 * st) for st in (h, h / 2)]
        _close(got["dalpha"].reshape(1), torch.tensor([(4 * da[1] - da[0]) / 3], dtype=f64), 1e-9,
               "dalpha vs finite differences")


def _autograd_forward(q, k, v, g, mu, alpha, w):
    """The operator in plain fp64 PyTorch ops, one token at a time (a second,
    separately written forward, differentiated by autograd)."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    S = torch.zeros(B, H, dk, dv, dtype=f64)
    ys = []
    for t in range(L):
        gam = torch.sigmoid(g[:, :, t])
        S = gam[..., None] * S + k[:, :, t, :, None] * v[:, :, t, None, :]
        yg = torch.einsum("bhi,bhij->bhj", q[:, :, t], S)
        lo = max(0, t - w + 1)
        kw, vw = k[:, :, lo:t + 1], v[:, :, lo:t + 1]
        a = torch.einsum("bhi,bhsi->bhs", q[:, :, t], kw)
        c = torch.einsum("bhi,hji->bhj", q[:, :, t], mu)
        logits = torch.cat([a, c], dim=-1)
        p = torch.softmax(logits, dim=-1)[..., : a.shape[-1]]
        ya = torch.einsum("bhs,bhsj->bhj", p, vw)
        ys.append(yg + alpha * ya)
    return torch.stack(ys, dim=2)


def pin_backward_vs_autograd(lib):
    # A longer sequence (crossing the oracle's internal checkpoints) against
    # autograd through the plain PyTorch forward above.
    B, H, L, d, w, m, alpha = 1, 2, 130, 8, 7, 3, 0.8
    q, k, v, g, mu = _qkvg(111, B, H, L, d, d, m=m, g_mean=1.0, g_std=2.0)
    dy = torch.randn(B, H, L, d, generator=_gen(112), dtype=f64)
    got = O.backward(q, k, v, g, mu, alpha, w, dy, lib=lib)
    leaves = [t.double().requires_grad_(True) for t in (q, k, v, g, mu)]
    al = torch.tensor(alpha, dtype=f64, requires_grad=True)
    y = _autograd_forward(*leaves, al, w)
    (y * dy).sum().backward()
    for name, t in zip(("dq", "dk", "dv", "dg", "dmu"), leaves):
        _close(got[name], t.grad, 1e-10, f"{name} vs autograd")
    _close(got["dalpha"].reshape(1), al.grad.reshape(1), 1e-10, "dalpha vs autograd")


def pin_backward_open_gates_have_no_gate_gradient(lib):
    # sigmoid(g) = 1 to fp64 precision (g = 1e4): the gate does not move, so
    # dg is exactly 0 whatever dy is.
    B, H, L, d = 1, 1, 20, 4
    q, k, v, g, mu = _qkvg(121, B, H, L, d, d, m=2)
    g = torch.full_like(g, 1e4)
    dy = torch.randn(B, H, L, d, generator=_gen(122), dtype=f64)
    got = O.backward(q, k, v, g, mu, 1.0, 4, dy, lib=lib)
    assert float(got["dg"].abs().max()) == 0.0
    assert float(got["dq"].abs().max()) > 0.0


# --- gate projection -----------------------------------------------------------

def pin_gate_projection_brute_force(lib):
    # Every output element by an explicit sum over the model dimension, with
    # the head-major placement g[b, h, t, i] <- row h * dk + i of W.
    B, L, dm, H, dk = 2, 3, 5, 2, 3
    gen = _gen(131)
    x = torch.randn(B, L, dm, generator=gen).to(torch.bfloat16)
    W = torch.randn(H * dk, dm, generator=gen).to(torch.bfloat16)
    got = O.gate_projection(x, W, H)
    assert tuple(got.shape) == (B, H, L, dk)
    for b in range(B):
        for h in range(H):
            for t in range(L):
                for i in range(dk):
                    ref = 0.0
                    for c in range(dm):
                        ref += float(x[b, t, c]) * float(W[h * dk + i, c])
                    assert abs(float(got[b, h, t, i]) - ref) <= 1e-12 * max(1.0, abs(ref)), (b, h, t, i)


PINS = [
    pin_log_sigmoid_vs_scipy,
    pin_recurrence_equals_product_form,
    pin_open_gates_are_causal_linear_attention,
    pin_constant_gate_geometric_form,
    pin_full_window_is_causal_softmax,
    pin_window_and_sinks_vs_masked_sdpa,
    pin_meta_logits_minus_inf_vanish,
    pin_single_token_closed_form,
    pin_linearity_in_alpha_and_v,
    pin_split_prefill_equals_whole,
    pin_decode_continues_prefill,
    pin_sink_free_weights_sum_to_one,
    pin_backward_vs_finite_differences,
    pin_backward_vs_autograd,
    pin_backward_open_gates_have_no_gate_gradient,
    pin_gate_projection_brute_force,
]
