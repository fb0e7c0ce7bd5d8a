"""Shared helpers of the GPU parity tests (device plumbing only)."""
from __future__ import annotations

import torch

from hybrid_gated_linear_attn_b300 import LizardState, lizard_attn_decode_step, lizard_attn_prefill
from hybrid_gated_linear_attn_b300 import build as B
from hybrid_gated_linear_attn_b300.inputs import rel_l2  # noqa: F401

TOL = {torch.float32: 1e-4, torch.bfloat16: 1e-2}


def ensure_built():
    B.build()


def to_dev(d: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def gpu_prefill(inp: dict, w: int, with_state: bool = True):
    """Run the CUDA prefill; returns y (CPU) and the state (device)."""
    q, k, v, g, mu = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu"))
    Bn, H, L, dk = q.shape
    st = LizardState(Bn, H, dk, v.shape[-1], w, dtype=q.dtype) if with_state else None
    y = lizard_attn_prefill(q, k, v, g, mu, inp["alpha"], w, state=st)
    torch.cuda.synchronize()
    return y.cpu(), st


def gpu_decode_step(step_inp: dict, mu, alpha, st: LizardState):
    q, k, v, g = (step_inp[n].cuda() for n in ("q", "k", "v", "g"))
    return lizard_attn_decode_step(q, k, v, g, mu.cuda(), alpha, st)
