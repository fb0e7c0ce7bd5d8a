"""Lizard hybrid attention operator (gated linear attention + anchor window
with meta-memory sinks) as hand-written CUDA for B300 (sm_103a), behind the
C ABI of ``include/lizard_attn.h``.
"""
from .lizard_attn import (  # noqa: F401
    LizardError,
    LizardState,
    lizard_attn_backward,
    lizard_attn_decode_step,
    lizard_attn_prefill,
    lizard_attn_prefill_continue,
    lizard_attn_prefill_noalloc,
    lizard_check_device_status,
    lizard_gate_projection,
    lizard_scratch_reserved,
    lizard_scratch_trim,
    lizard_state_init,
    lizard_status_string,
)
