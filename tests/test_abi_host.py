"""Host-side checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments with the documented status
codes before launching anything.

Every call below carries at least one invalid argument (or is an empty
B == 0 call), so no kernel is ever launched with the fake pointers used here;
that keeps these tests safe on a machine with a GPU as well.
"""
import ctypes
import os
import re

import pytest

from hybrid_gated_linear_attn_b300 import build as B
from hybrid_gated_linear_attn_b300 import lizard_attn as LA

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lizard_attn.h")

OK, INVALID, UNSUPPORTED = LA.LIZARD_OK, LA.LIZARD_ERR_INVALID_ARG, LA.LIZARD_ERR_UNSUPPORTED
A = 0x7f0000000000          # a 16-byte aligned fake device address (never dereferenced)
MIS = A + 8                 # misaligned


@pytest.fixture(scope="module")
def lib():
    B.build()
    return LA.library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"LIZARD_API\s+[^;(]*?\b(lizard_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(LA.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert LA.lizard_status_string(OK) == "LIZARD_OK"
    assert LA.lizard_status_string(INVALID) == "LIZARD_ERR_INVALID_ARG"
    assert LA.lizard_status_string(UNSUPPORTED) == "LIZARD_ERR_UNSUPPORTED"
    assert LA.lizard_status_string(LA.LIZARD_ERR_CUDA) == "LIZARD_ERR_CUDA"
    assert LA.lizard_status_string(LA.LIZARD_ERR_TIMEOUT) == "LIZARD_ERR_TIMEOUT"
    assert LA.lizard_status_string(99) == "LIZARD_ERR_UNKNOWN"


def prefill(lib, q=A, k=A, v=A, g=A, mu=A, alpha=1.0, Bn=2, H=4, L=128, dk=128, dv=128, w=64, m=4,
            dtype=LA.LIZARD_BF16, y=A, st=None):
    return lib.lizard_attn_prefill(q, k, v, g, mu, alpha, Bn, H, L, dk, dv, w, m, dtype, y,
                                   ctypes.byref(st) if st is not None else None, None)


def state(S=A, rk=A, rv=A, pos=A, Bn=2, H=4, dk=128, dv=128, w=64, dtype=LA.LIZARD_BF16):
    return LA.lizard_state(S, rk, rv, pos, Bn, H, dk, dv, w, dtype)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(k=None), INVALID), (dict(v=None), INVALID), (dict(g=None), INVALID),
    (dict(y=None), INVALID), (dict(mu=None), INVALID),
    (dict(q=MIS), INVALID), (dict(y=MIS), INVALID), (dict(mu=MIS), INVALID),
    (dict(dtype=7), INVALID), (dict(w=0), INVALID), (dict(w=-3), INVALID), (dict(m=-1), INVALID),
    (dict(L=-1), INVALID), (dict(H=0), INVALID), (dict(Bn=-1), INVALID), (dict(dk=0), INVALID),
    (dict(dk=96, dv=96), UNSUPPORTED), (dict(dk=128, dv=64), UNSUPPORTED), (dict(dk=512, dv=512), UNSUPPORTED),
    (dict(w=LA.LIZARD_MAX_WINDOW + 1), UNSUPPORTED), (dict(m=LA.LIZARD_MAX_META + 1), UNSUPPORTED),
])
def test_prefill_rejects(lib, kw, code):
    assert prefill(lib, **kw) == code


def test_prefill_meta_may_be_null_when_m_is_zero(lib):
    # m == 0 with a null meta pointer is valid; w = 0 keeps the call from launching.
    assert prefill(lib, mu=None, m=0, w=0) == INVALID
    assert prefill(lib, mu=None, m=0, Bn=0) == OK


def test_empty_batch_is_ok_without_launch(lib):
    assert prefill(lib, Bn=0) == OK


def test_empty_prompt_may_pass_null_token_pointers(lib):
    # L == 0: null q/k/v/g/y are accepted; w = 0 still stops it before launch.
    assert prefill(lib, q=None, k=None, v=None, g=None, y=None, L=0, w=0) == INVALID
    assert prefill(lib, q=None, k=None, v=None, g=None, y=None, L=0, Bn=0) == OK
    assert prefill(lib, q=None, L=1, Bn=0) == INVALID


@pytest.mark.parametrize("skw,code", [
    (dict(S=None), INVALID), (dict(rk=None), INVALID), (dict(rv=None), INVALID), (dict(pos=None), INVALID),
    (dict(S=MIS), INVALID), (dict(pos=A + 4), INVALID),
    (dict(Bn=3), INVALID), (dict(H=5), INVALID), (dict(w=32), INVALID), (dict(dtype=LA.LIZARD_F32), INVALID),
    (dict(dk=64, dv=64), INVALID),
])
def test_prefill_state_mismatch(lib, skw, code):
    # The call itself is valid except for the state; w=64 matches the default.
    # Each case is rejected before launch.
    assert prefill(lib, st=state(**skw)) == code


def decode(lib, q=A, k=A, v=A, g=A, mu=A, alpha=1.0, m=4, y=A, st="default"):
    st = state() if st == "default" else st
    return lib.lizard_attn_decode_step(q, k, v, g, mu, alpha, m, y,
                                       ctypes.byref(st) if st is not None else None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(v=None), INVALID), (dict(y=None), INVALID), (dict(mu=None), INVALID),
    (dict(g=MIS), INVALID), (dict(m=-1), INVALID), (dict(m=LA.LIZARD_MAX_META + 1), UNSUPPORTED),
    (dict(st=None), INVALID),
    (dict(st=state(w=0)), INVALID), (dict(st=state(H=0)), INVALID), (dict(st=state(dtype=5)), INVALID),
    (dict(st=state(dk=96, dv=96)), UNSUPPORTED), (dict(st=state(w=LA.LIZARD_MAX_WINDOW + 1)), UNSUPPORTED),
    (dict(st=state(S=None)), INVALID), (dict(st=state(rk=MIS)), INVALID),
    # d = 256 in fp32 stages ring and meta keys in shared memory: w = 100 with
    # 16 meta keys does not fit (checked on the host, before any launch)
    (dict(st=state(dk=256, dv=256, w=100, dtype=LA.LIZARD_F32), m=16), UNSUPPORTED),
    (dict(st=state(H=1 << 20)), UNSUPPORTED),
])
def test_decode_rejects(lib, kw, code):
    assert decode(lib, **kw) == code


def test_state_init_rejects(lib):
    assert lib.lizard_state_init(None, None) == INVALID
    for bad in (state(S=None), state(pos=A + 4), state(w=0), state(dtype=9)):
        assert lib.lizard_state_init(ctypes.byref(bad), None) == INVALID
    assert lib.lizard_state_init(ctypes.byref(state(dk=80, dv=80)), None) == UNSUPPORTED
    assert lib.lizard_state_init(ctypes.byref(state(Bn=0)), None) == OK


def test_binding_names_match_the_c_abi():
    import hybrid_gated_linear_attn_b300 as pkg
    for name in ("lizard_state_init", "lizard_attn_prefill", "lizard_attn_prefill_continue", "lizard_attn_prefill_noalloc",
                 "lizard_attn_backward", "lizard_gate_projection",
                 "lizard_attn_decode_step", "lizard_check_device_status", "lizard_status_string",
                 "lizard_scratch_trim", "lizard_scratch_reserved"):
        assert callable(getattr(pkg, name))


def cont(lib, q=A, k=A, v=A, g=A, mu=A, alpha=1.0, L=128, m=4, y=A, st="default"):
    st = state() if st == "default" else st
    return lib.lizard_attn_prefill_continue(q, k, v, g, mu, alpha, L, m, y,
                                            ctypes.byref(st) if st is not None else None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(k=None), INVALID), (dict(g=None), INVALID), (dict(y=None), INVALID),
    (dict(mu=None), INVALID), (dict(v=MIS), INVALID), (dict(mu=MIS), INVALID),
    (dict(L=-1), INVALID), (dict(m=-1), INVALID), (dict(m=LA.LIZARD_MAX_META + 1), UNSUPPORTED),
    (dict(st=None), INVALID), (dict(st=state(pos=None)), INVALID), (dict(st=state(S=MIS)), INVALID),
    (dict(st=state(w=0)), INVALID), (dict(st=state(dtype=3)), INVALID),
    (dict(st=state(dk=96, dv=96)), UNSUPPORTED), (dict(st=state(w=LA.LIZARD_MAX_WINDOW + 1)), UNSUPPORTED),
])
def test_continue_rejects(lib, kw, code):
    assert cont(lib, **kw) == code


def test_continue_empty_calls_launch_nothing(lib):
    # No new token, or no sequence: the state stays as it is and nothing runs.
    assert cont(lib, q=None, k=None, v=None, g=None, y=None, L=0) == OK
    assert cont(lib, st=state(Bn=0)) == OK


def backward(lib, q=A, k=A, v=A, g=A, mu=A, alpha=1.0, Bn=2, H=4, L=128, dk=128, dv=128, w=64, m=4,
             dtype=LA.LIZARD_BF16, dy=A, dq=A, dko=A, dvo=A, dg=A, dmu=A, dal=A):
    return lib.lizard_attn_backward(q, k, v, g, mu, alpha, Bn, H, L, dk, dv, w, m, dtype, dy, dq, dko, dvo, dg,
                                    dmu, dal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), INVALID), (dict(dy=None), INVALID), (dict(dq=None), INVALID), (dict(dg=None), INVALID),
    (dict(dvo=None), INVALID), (dict(mu=None), INVALID), (dict(dmu=None), INVALID), (dict(dal=None), INVALID),
    (dict(dal=A + 2), INVALID), (dict(dy=MIS), INVALID), (dict(dmu=MIS), INVALID),
    (dict(dtype=7), INVALID), (dict(w=0), INVALID), (dict(m=-1), INVALID), (dict(L=-1), INVALID),
    (dict(H=0), INVALID), (dict(dk=96, dv=96), UNSUPPORTED), (dict(dk=128, dv=64), UNSUPPORTED),
    (dict(dk=256, dv=256), UNSUPPORTED),  # the backward is built for d in {64, 128}
    (dict(w=LA.LIZARD_MAX_WINDOW + 1), UNSUPPORTED), (dict(m=LA.LIZARD_MAX_META + 1), UNSUPPORTED),
])
def test_backward_rejects(lib, kw, code):
    assert backward(lib, **kw) == code


def gproj(lib, x=A, w=A, Bn=2, L=128, dm=256, H=4, dk=128, dtype=LA.LIZARD_BF16, g=A):
    return lib.lizard_gate_projection(x, w, Bn, L, dm, H, dk, dtype, g, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), INVALID), (dict(w=None), INVALID), (dict(g=None), INVALID), (dict(x=MIS), INVALID),
    (dict(dtype=9), INVALID), (dict(Bn=-1), INVALID), (dict(dm=0), INVALID), (dict(H=0), INVALID),
    (dict(dk=64), UNSUPPORTED), (dict(dtype=LA.LIZARD_F32), UNSUPPORTED), (dict(dm=100), UNSUPPORTED),
])
def test_gate_projection_rejects(lib, kw, code):
    assert gproj(lib, **kw) == code


def test_gate_projection_empty_is_ok(lib):
    assert gproj(lib, x=None, w=None, g=None, L=0) == OK


def variant(alpha_h=None, Hkv=0):
    return ctypes.byref(LA.lizard_variant(alpha_h, Hkv))


@pytest.mark.parametrize("var,code", [
    (dict(Hkv=3), INVALID),          # does not divide H = 4
    (dict(Hkv=-1), INVALID),
    (dict(Hkv=5), INVALID),          # more key/value heads than query heads
    (dict(alpha_h=A + 2), INVALID),  # misaligned per-head weights
])
def test_variant_rejected_by_every_entry_point(lib, var, code):
    v = variant(**var)
    assert lib.lizard_attn_prefill_v(A, A, A, A, A, 1.0, 2, 4, 128, 128, 128, 64, 4, LA.LIZARD_BF16, A,
                                     None, v, None) == code
    st = state()
    assert lib.lizard_attn_prefill_continue_v(A, A, A, A, A, 1.0, 128, 4, A, ctypes.byref(st), v, None) == code
    assert lib.lizard_attn_decode_step_v(A, A, A, A, A, 1.0, 4, A, ctypes.byref(st), v, None) == code
    assert lib.lizard_attn_backward_v(A, A, A, A, A, 1.0, 2, 4, 128, 128, 128, 64, 4, LA.LIZARD_BF16, A, A, A, A, A,
                                      A, A, v, None) == code


def test_valid_variant_on_empty_calls_launches_nothing(lib):
    v = variant(alpha_h=A, Hkv=2)
    assert lib.lizard_attn_prefill_v(A, A, A, A, A, 1.0, 0, 4, 128, 128, 128, 64, 4, LA.LIZARD_BF16, A,
                                     None, v, None) == OK
    assert lib.lizard_attn_prefill_continue_v(None, None, None, None, A, 1.0, 0, 4, None,
                                              ctypes.byref(state()), v, None) == OK


def noalloc(lib, q=A, k=A, v=A, g=A, mu=A, alpha=1.0, Bn=2, H=4, L=128, dk=128, dv=128, w=64, m=4,
            dtype=LA.LIZARD_BF16, y=A, st=None):
    return lib.lizard_attn_prefill_noalloc(q, k, v, g, mu, alpha, Bn, H, L, dk, dv, w, m, dtype, y,
                                           ctypes.byref(st) if st is not None else None, None)


@pytest.mark.parametrize("kw,code", [
    # the allocation-free call covers the bf16 tensor-core prefill only: d = 128 or 64
    (dict(dtype=LA.LIZARD_F32), UNSUPPORTED),
    (dict(dk=64, dv=128), UNSUPPORTED), (dict(dk=96, dv=96), UNSUPPORTED), (dict(w=129), UNSUPPORTED),
    (dict(m=LA.LIZARD_MAX_META + 1), UNSUPPORTED), (dict(dk=256, dv=256, st=state(dk=256, dv=256)), UNSUPPORTED),
    (dict(q=None), INVALID), (dict(g=None), INVALID), (dict(y=None), INVALID), (dict(mu=None), INVALID),
    (dict(v=MIS), INVALID), (dict(y=MIS), INVALID), (dict(dtype=7), INVALID), (dict(w=0), INVALID),
    (dict(m=-1), INVALID), (dict(L=-1), INVALID), (dict(H=0), INVALID), (dict(Bn=-1), INVALID),
    (dict(st=state(Bn=3)), INVALID), (dict(st=state(w=32)), INVALID), (dict(st=state(S=None)), INVALID),
    (dict(st=state(pos=A + 4)), INVALID), (dict(st=state(dtype=LA.LIZARD_F32)), INVALID),
])
def test_noalloc_rejects(lib, kw, code):
    assert noalloc(lib, **kw) == code


def test_noalloc_empty_calls_launch_nothing(lib):
    assert noalloc(lib, Bn=0) == OK
    assert noalloc(lib, q=None, k=None, v=None, g=None, y=None, L=0) == OK  # no state: nothing to reset


def test_state_batch_view_shares_the_buffers():
    """LizardState.batch(b0, b1) is a view of sequences b0 .. b1-1: the
    struct it hands to the C ABI points into the parent's buffers."""
    st = LA.LizardState(4, 2, 64, 64, 16, device="cpu")
    v = st.batch(1, 3)
    assert (v.B, v.H, v.dk, v.dv, v.w) == (2, 2, 64, 64, 16)
    c = v.c_struct()
    assert c.S == st.S[1].data_ptr() and c.pos == st.pos[1].data_ptr()
    assert c.ring_k == st.ring_k[1].data_ptr() and c.ring_v == st.ring_v[1].data_ptr()
    assert c.B == 2
    with pytest.raises(ValueError):
        st.batch(3, 3)
    with pytest.raises(ValueError):
        st.batch(2, 5)


def test_state_pos_needs_only_8_byte_alignment(lib):
    """pos of a batch slice (pos + b0) is only 8-byte aligned, and valid.
    With B = 0 nothing is launched, so the fake addresses stay untouched."""
    st = state(pos=A + 8, Bn=0)
    assert lib.lizard_state_init(ctypes.byref(st), None) == LA.LIZARD_OK
