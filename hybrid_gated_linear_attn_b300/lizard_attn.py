"""Python binding of ``liblizard_attn.so`` (ctypes; argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors that already live on the GPU.  Every step of the operator runs in the
library's CUDA kernels; there is no Python or CPU fallback: if the library is
missing or cannot be loaded, the first call raises.

The C contract (layouts, alignment, errors) is in ``include/lizard_attn.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "liblizard_attn.so")

LIZARD_OK, LIZARD_ERR_INVALID_ARG, LIZARD_ERR_UNSUPPORTED, LIZARD_ERR_CUDA, LIZARD_ERR_TIMEOUT = range(5)
LIZARD_F32, LIZARD_BF16 = 0, 1
LIZARD_MAX_WINDOW = 128
LIZARD_MAX_META = 16

EXPORTS = ("lizard_state_init", "lizard_attn_prefill", "lizard_attn_prefill_v", "lizard_attn_prefill_continue",
           "lizard_attn_prefill_continue_v", "lizard_attn_prefill_noalloc", "lizard_attn_backward",
           "lizard_attn_backward_v", "lizard_gate_projection", "lizard_attn_decode_step", "lizard_attn_decode_step_v",
           "lizard_check_device_status", "lizard_status_string", "lizard_scratch_trim", "lizard_scratch_reserved")


class LizardError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)}")


class lizard_variant(ctypes.Structure):
    _fields_ = [("alpha_h", ctypes.c_void_p), ("Hkv", ctypes.c_int)]


def _variant(alpha_h=None, Hkv=0):
    """A lizard_variant by reference, or None for the plain operator."""
    if alpha_h is None and not Hkv:
        return None
    return ctypes.byref(lizard_variant(alpha_h.data_ptr() if alpha_h is not None else None, int(Hkv)))


class lizard_state(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("ring_k", ctypes.c_void_p), ("ring_v", ctypes.c_void_p),
                ("pos", ctypes.c_void_p), ("B", ctypes.c_int), ("H", ctypes.c_int), ("dk", ctypes.c_int),
                ("dv", ctypes.c_int), ("w", ctypes.c_int), ("dtype", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (once) and declare the C signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"liblizard_attn.so not built ({path}); run "
                               "`python -m hybrid_gated_linear_attn_b300.build`")
        lib = ctypes.CDLL(path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        SP = ctypes.POINTER(lizard_state)
        lib.lizard_state_init.argtypes = [SP, P]
        lib.lizard_state_init.restype = I
        VP = ctypes.POINTER(lizard_variant)
        lib.lizard_attn_prefill.argtypes = [P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, SP, P]
        lib.lizard_attn_prefill.restype = I
        lib.lizard_attn_prefill_v.argtypes = [P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, SP, VP, P]
        lib.lizard_attn_prefill_v.restype = I
        lib.lizard_attn_prefill_continue_v.argtypes = [P, P, P, P, P, F, I, I, P, SP, VP, P]
        lib.lizard_attn_prefill_continue_v.restype = I
        lib.lizard_attn_backward_v.argtypes = [P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, VP, P]
        lib.lizard_attn_backward_v.restype = I
        lib.lizard_attn_decode_step_v.argtypes = [P, P, P, P, P, F, I, P, SP, VP, P]
        lib.lizard_attn_decode_step_v.restype = I
        lib.lizard_attn_prefill_continue.argtypes = [P, P, P, P, P, F, I, I, P, SP, P]
        lib.lizard_attn_prefill_continue.restype = I
        lib.lizard_attn_prefill_noalloc.argtypes = [P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, SP, P]
        lib.lizard_attn_prefill_noalloc.restype = I
        lib.lizard_attn_backward.argtypes = [P, P, P, P, P, F, I, I, I, I, I, I, I, I, P, P, P, P, P, P, P, P]
        lib.lizard_attn_backward.restype = I
        lib.lizard_gate_projection.argtypes = [P, P, I, I, I, I, I, I, P, P]
        lib.lizard_gate_projection.restype = I
        lib.lizard_attn_decode_step.argtypes = [P, P, P, P, P, F, I, P, SP, P]
        lib.lizard_attn_decode_step.restype = I
        lib.lizard_check_device_status.argtypes = [P]
        lib.lizard_check_device_status.restype = I
        lib.lizard_status_string.argtypes = [I]
        lib.lizard_status_string.restype = ctypes.c_char_p
        lib.lizard_scratch_trim.argtypes = [ctypes.c_size_t]
        lib.lizard_scratch_trim.restype = I
        lib.lizard_scratch_reserved.argtypes = [ctypes.POINTER(ctypes.c_size_t)]
        lib.lizard_scratch_reserved.restype = I
        _lib = lib
        return lib


def status_name(status: int) -> str:
    try:
        return library().lizard_status_string(int(status)).decode()
    except Exception:  # library missing: still give a readable name
        return f"status {status}"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LIZARD_F32
    if t.dtype == torch.bfloat16:
        return LIZARD_BF16
    raise TypeError(f"lizard_attn takes fp32 or bf16 tensors, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _check(rc: int, where: str):
    if rc != LIZARD_OK:
        raise LizardError(rc, where)


class LizardState:
    """Caller-owned device buffers of the recurrent state (S, ring, pos)."""

    def __init__(self, B, H, dk, dv, w, dtype=torch.bfloat16, device="cuda"):
        self.B, self.H, self.dk, self.dv, self.w, self.dtype = B, H, dk, dv, w, dtype
        self.S = torch.empty(B, H, dk, dv, dtype=torch.float32, device=device)
        self.ring_k = torch.empty(B, H, w, dk, dtype=dtype, device=device)
        self.ring_v = torch.empty(B, H, w, dv, dtype=dtype, device=device)
        self.pos = torch.empty(B, dtype=torch.int64, device=device)

    def batch(self, b0: int, b1: int) -> "LizardState":
        """The state of sequences b0 .. b1-1: a view on the same buffers (the
        batch is the outermost dim of every buffer), for calls on a slice of
        the batch."""
        if not 0 <= b0 < b1 <= self.B:
            raise ValueError(f"batch slice {b0}:{b1} of {self.B}")
        view = object.__new__(LizardState)
        view.B, view.H, view.dk, view.dv, view.w, view.dtype = b1 - b0, self.H, self.dk, self.dv, self.w, self.dtype
        view.S, view.ring_k, view.ring_v, view.pos = self.S[b0:b1], self.ring_k[b0:b1], self.ring_v[b0:b1], self.pos[b0:b1]
        return view

    def c_struct(self) -> lizard_state:
        return lizard_state(self.S.data_ptr(), self.ring_k.data_ptr(), self.ring_v.data_ptr(),
                            self.pos.data_ptr(), self.B, self.H, self.dk, self.dv, self.w,
                            LIZARD_F32 if self.dtype == torch.float32 else LIZARD_BF16)


def lizard_state_init(state: LizardState, stream=None) -> LizardState:
    st = state.c_struct()
    _check(library().lizard_state_init(ctypes.byref(st), _stream(stream)), "lizard_state_init")
    return state


def lizard_attn_prefill(q, k, v, g, meta_k, alpha, w, y=None, state: LizardState | None = None,
                        stream=None, alpha_h=None, Hkv=0) -> torch.Tensor:
    """y = Lizard(q, k, v, g; meta_k, alpha, w) over [B,H,L,d] tensors.

    ``state``, when given, receives the state after the prompt.  ``alpha_h``
    (a [H] fp32 device tensor) and ``Hkv`` select the variants of
    ``lizard_variant`` (k, v then [B,Hkv,L,d]).
    """
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    m = meta_k.shape[1] if meta_k is not None else 0
    if y is None:
        y = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    st = state.c_struct() if state is not None else None
    rc = library().lizard_attn_prefill_v(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(meta_k) if m > 0 else None, float(alpha),
        B, H, L, dk, dv, int(w), m, _dtype_code(q), _ptr(y),
        ctypes.byref(st) if st is not None else None, _variant(alpha_h, Hkv), _stream(stream))
    _check(rc, "lizard_attn_prefill")
    return y


def lizard_attn_prefill_continue(q, k, v, g, meta_k, alpha, state: LizardState, y=None,
                                 stream=None, alpha_h=None, Hkv=0) -> torch.Tensor:
    """L more tokens per sequence ([B,H,L,d] tensors), continuing from
    ``state`` (updated in place): the window and the gate state carry on
    from the tokens the state has already consumed."""
    L = q.shape[2]
    m = meta_k.shape[1] if meta_k is not None else 0
    if y is None:
        y = torch.empty(state.B, state.H, L, state.dv, dtype=q.dtype, device=q.device)
    st = state.c_struct()
    rc = library().lizard_attn_prefill_continue_v(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(meta_k) if m > 0 else None, float(alpha), L, m,
        _ptr(y), ctypes.byref(st), _variant(alpha_h, Hkv), _stream(stream))
    _check(rc, "lizard_attn_prefill_continue")
    return y


def lizard_attn_prefill_noalloc(q, k, v, g, meta_k, alpha, w, y=None, state: LizardState | None = None,
                                stream=None) -> torch.Tensor:
    """lizard_attn_prefill without device allocation inside the call (bf16,
    d = 128, w <= 65): segment states go to the library's fixed device array.
    ``y`` is allocated here when not given; pass it to allocate nothing."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    m = meta_k.shape[1] if meta_k is not None else 0
    if y is None:
        y = torch.empty(B, H, L, dv, dtype=q.dtype, device=q.device)
    st = state.c_struct() if state is not None else None
    rc = library().lizard_attn_prefill_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(meta_k) if m > 0 else None, float(alpha),
        B, H, L, dk, dv, int(w), m, _dtype_code(q), _ptr(y),
        ctypes.byref(st) if st is not None else None, _stream(stream))
    _check(rc, "lizard_attn_prefill_noalloc")
    return y


def lizard_attn_backward(q, k, v, g, meta_k, alpha, w, dy, stream=None, alpha_h=None, Hkv=0):
    """Gradients of sum(dy * y) through the operator over [B,H,L,d] tensors
    that start from the empty state.  Returns (dq, dk, dv, dg, dmeta_k,
    dalpha): the first four in the input dtype, dmeta_k [H,m,dk] fp32 (None
    when m == 0) and dalpha a 0-d fp32 tensor, all on the inputs' device."""
    B, H, L, dk = q.shape
    dv = v.shape[-1]
    m = meta_k.shape[1] if meta_k is not None else 0
    dq, dg = torch.empty_like(q), torch.empty_like(g)
    dk_, dv_ = torch.empty_like(k), torch.empty_like(v)
    dmeta = torch.empty(H, m, dk, dtype=torch.float32, device=q.device) if m > 0 else None
    dalpha = torch.empty((H,) if alpha_h is not None else (), dtype=torch.float32, device=q.device)
    rc = library().lizard_attn_backward_v(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(meta_k) if m > 0 else None, float(alpha),
        B, H, L, dk, dv, int(w), m, _dtype_code(q), _ptr(dy), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg),
        _ptr(dmeta) if m > 0 else None, _ptr(dalpha), _variant(alpha_h, Hkv), _stream(stream))
    _check(rc, "lizard_attn_backward")
    return dq, dk_, dv_, dg, dmeta, dalpha


def lizard_gate_projection(x, w_gamma, H, g=None, stream=None) -> torch.Tensor:
    """Gate logits g [B, H, L, dk] (head-major) = x [B, L, dmodel] times the
    gate weight w_gamma [H * dk, dmodel] transposed."""
    B, L, dmodel = x.shape
    dk = w_gamma.shape[0] // H
    if g is None:
        g = torch.empty(B, H, L, dk, dtype=x.dtype, device=x.device)
    rc = library().lizard_gate_projection(_ptr(x), _ptr(w_gamma), B, L, dmodel, H, dk, _dtype_code(x), _ptr(g),
                                          _stream(stream))
    _check(rc, "lizard_gate_projection")
    return g


def lizard_attn_decode_step(q, k, v, g, meta_k, alpha, state: LizardState, y=None, stream=None,
                            alpha_h=None, Hkv=0) -> torch.Tensor:
    """One token per sequence: q,k,g [B,H,dk], v [B,H,dv] -> y [B,H,dv]."""
    m = meta_k.shape[1] if meta_k is not None else 0
    if y is None:
        y = torch.empty(state.B, state.H, state.dv, dtype=q.dtype, device=q.device)
    st = state.c_struct()
    rc = library().lizard_attn_decode_step_v(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(meta_k) if m > 0 else None, float(alpha), m,
        _ptr(y), ctypes.byref(st), _variant(alpha_h, Hkv), _stream(stream))
    _check(rc, "lizard_attn_decode_step")
    return y


def lizard_check_device_status(stream=None) -> None:
    _check(library().lizard_check_device_status(_stream(stream)), "lizard_check_device_status")


def lizard_status_string(status: int) -> str:
    return library().lizard_status_string(int(status)).decode()


def lizard_scratch_trim(keep_bytes: int = 0) -> None:
    """Hand the library's scratch on the current device back to the driver,
    keeping at most ``keep_bytes`` (synchronise earlier calls first)."""
    _check(library().lizard_scratch_trim(int(keep_bytes)), "lizard_scratch_trim")


def lizard_scratch_reserved() -> int:
    """Bytes the library's scratch pool holds on the current device."""
    n = ctypes.c_size_t(0)
    _check(library().lizard_scratch_reserved(ctypes.byref(n)), "lizard_scratch_reserved")
    return int(n.value)
