"""Seeded synthetic inputs for the Lizard hybrid attention operator.

This module only draws random tensors with the shapes and distributions of
the workloads below.  It holds none of the operator's arithmetic, so the
CUDA path and the CPU oracle can both consume its output without sharing any
of the method's code.

All tensors are drawn on the CPU with ``torch.Generator().manual_seed``, in
fp32, then cast to the workload's storage dtype, so every consumer sees the
same bits.  Layout is head-major: q, k, g are [B, H, L, d_k], v is
[B, H, L, d_v], meta keys are [H, m, d_k].

Workloads (the Lizard pages evaluate Llama-3-8B and Mistral-7B layers; the
shapes below stand in for those layers with random data):

* ``tiny_f32``      B1 H2 L256 d64, fp32, g~N(3,1), w16 m4 alpha 0.5, seed 0
* ``llama3_8b``     B4 H32 L4096 d128, bf16, g~N(3,1), w64 m4 alpha 1.0
* ``decay_stress``  B2 H32 L8192 d128, bf16, g~N(0,2), w128 m8 alpha 0.5
* ``decode``        64 sequences x H32 d128 bf16, fp32 state ~N(0,1)/128,
                    full w=64 ring, m4, 1024 steps of q,k,v,g as llama3_8b
* ``long_context``  B1 H32 L65536 d128, bf16, g~N(4,1), w64 m4 alpha 1.0,
                    then 128 decode steps

q and k are N(0,1) scaled by 1/sqrt(d_k); v is N(0,1); meta keys are
N(0,1)/8; gate logits are N(g_mean, g_std) per (token, head, key dim).
"""
from __future__ import annotations

import dataclasses
import math

import torch

F32 = "f32"
BF16 = "bf16"


def torch_dtype(dt: str) -> torch.dtype:
    return {F32: torch.float32, BF16: torch.bfloat16}[dt]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    dk: int
    dv: int
    w: int
    m: int
    alpha: float
    dtype: str
    g_mean: float
    g_std: float
    seed: int
    decode_steps: int = 0

    @property
    def qk_scale(self) -> float:
        return 1.0 / math.sqrt(self.dk)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 2, 256, 64, 64, 16, 4, 0.5, F32, 3.0, 1.0, 0),
    "llama3_8b": Workload("llama3_8b", 4, 32, 4096, 128, 128, 64, 4, 1.0, BF16, 3.0, 1.0, 1),
    "decay_stress": Workload("decay_stress", 2, 32, 8192, 128, 128, 128, 8, 0.5, BF16, 0.0, 2.0, 2),
    # The decode workload: B is the number of sequences, L the ring history
    # already consumed (a full ring), decode_steps the tokens generated.
    "decode": Workload("decode", 64, 32, 64, 128, 128, 64, 4, 1.0, BF16, 3.0, 1.0, 3, decode_steps=1024),
    "long_context": Workload("long_context", 1, 32, 65536, 128, 128, 64, 4, 1.0, BF16, 4.0, 1.0, 4,
                             decode_steps=128),
    # head dim 64 (a Llama-3.2-1B-shaped layer: 32 heads of 64), otherwise
    # the headline prefill's recipe
    "d64": Workload("d64", 4, 32, 4096, 64, 64, 64, 4, 1.0, BF16, 3.0, 1.0, 5),
}


def _randn(gen: torch.Generator, shape, scale: float = 1.0, mean: float = 0.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    if mean != 0.0:
        x.add_(mean)
    return x


def prefill_inputs(wl: Workload, L: int | None = None, seed: int | None = None) -> dict:
    """q, k, v, g [B,H,L,d], meta keys mu [H,m,dk] and alpha for a prefill.

    ``L`` overrides the sequence length (same distributions); ``seed``
    overrides the workload's seed.
    """
    L = wl.L if L is None else L
    gen = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    dt = torch_dtype(wl.dtype)
    B, H = wl.B, wl.H
    q = _randn(gen, (B, H, L, wl.dk), wl.qk_scale).to(dt)
    k = _randn(gen, (B, H, L, wl.dk), wl.qk_scale).to(dt)
    v = _randn(gen, (B, H, L, wl.dv)).to(dt)
    g = _randn(gen, (B, H, L, wl.dk), wl.g_std, wl.g_mean).to(dt)
    mu = _randn(gen, (H, wl.m, wl.dk), 1.0 / 8.0).to(dt)
    return dict(q=q, k=k, v=v, g=g, mu=mu, alpha=wl.alpha)


def decode_initial_state(wl: Workload, seed: int | None = None) -> dict:
    """Given-history state for the decode workload.

    S [B,H,dk,dv] fp32 ~ N(0,1)/128; the ring holds ``wl.L`` tokens of k, v
    drawn like the prefill inputs (a full ring when wl.L >= wl.w); pos = wl.L.
    Ring slot of token p is p mod w.  Also returns the history as plain
    [B,H,hist,d] tensors (oldest first) and meta keys mu.
    """
    gen = torch.Generator().manual_seed((wl.seed if seed is None else seed) * 7919 + 17)
    dt = torch_dtype(wl.dtype)
    B, H, w = wl.B, wl.H, wl.w
    S = _randn(gen, (B, H, wl.dk, wl.dv), 1.0 / 128.0)
    hist = wl.L
    hk = _randn(gen, (B, H, hist, wl.dk), wl.qk_scale).to(dt)
    hv = _randn(gen, (B, H, hist, wl.dv)).to(dt)
    mu = _randn(gen, (H, wl.m, wl.dk), 1.0 / 8.0).to(dt)
    ring_k = torch.zeros((B, H, w, wl.dk), dtype=dt)
    ring_v = torch.zeros((B, H, w, wl.dv), dtype=dt)
    for p in range(max(0, hist - w), hist):
        ring_k[:, :, p % w] = hk[:, :, p]
        ring_v[:, :, p % w] = hv[:, :, p]
    pos = torch.full((B,), hist, dtype=torch.int64)
    return dict(S=S, ring_k=ring_k, ring_v=ring_v, pos=pos, hist_k=hk, hist_v=hv, mu=mu)


def decode_step_inputs(wl: Workload, step: int, seed: int | None = None) -> dict:
    """q, k, v, g [B,H,d] for decode step ``step`` (each step its own seed)."""
    base = wl.seed if seed is None else seed
    gen = torch.Generator().manual_seed(base * 1_000_003 + 101 + step)
    dt = torch_dtype(wl.dtype)
    B, H = wl.B, wl.H
    q = _randn(gen, (B, H, wl.dk), wl.qk_scale).to(dt)
    k = _randn(gen, (B, H, wl.dk), wl.qk_scale).to(dt)
    v = _randn(gen, (B, H, wl.dv)).to(dt)
    g = _randn(gen, (B, H, wl.dk), wl.g_std, wl.g_mean).to(dt)
    return dict(q=q, k=k, v=v, g=g)


def rel_l2(x: torch.Tensor, ref: torch.Tensor) -> float:
    """||x - ref||_2 / ||ref||_2 over all elements, in fp64."""
    x = x.double()
    ref = ref.double()
    return float(torch.linalg.vector_norm(x - ref) / torch.linalg.vector_norm(ref))


def gate_projection_inputs(B: int, L: int, dmodel: int, H: int, dk: int, seed: int = 5) -> dict:
    """Layer input x [B, L, dmodel] ~ N(0, 1) and gate weight W [H dk, dmodel]
    ~ N(0, 1) / sqrt(dmodel) (so the logits are ~N(0, 1)), both bf16."""
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(B, L, dmodel, generator=gen).to(torch.bfloat16)
    W = (torch.randn(H * dk, dmodel, generator=gen) / math.sqrt(dmodel)).to(torch.bfloat16)
    return {"x": x, "W": W}
