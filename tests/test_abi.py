"""The C ABI without a GPU: the library loads, exports what include/sla.h
declares, and rejects bad arguments before it touches CUDA."""
import ctypes
import os
import re

import pytest

from gated_linear_attention_attn_b300 import build

build.build()
from gated_linear_attention_attn_b300 import sla  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "sla.h")

# Fake device addresses: the checks below fail before any CUDA call, so the
# library never dereferences them.
A = 0x10000000
STEP = 0x01000000


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert set(_declared_functions()) == set(sla.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(sla.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    assert sla.status_string(sla.OK) == "ok"
    assert "argument" in sla.status_string(sla.INVALID_ARG)
    assert "timed out" in sla.status_string(sla.DEVICE_TIMEOUT)
    assert sla.status_string(99) == "unknown status"


def _fwd(q=A, k=A + STEP, v=A + 2 * STEP, g=A + 3 * STEP, out=A + 4 * STEP, B=1, H=2, N=256,
         d=128, rope=None, eps=1e-6, f32=False):
    fn = sla.raw_lib().sla_linattn_forward_f32 if f32 else sla.raw_lib().sla_linattn_forward
    r = ctypes.byref(rope) if rope is not None else None
    return fn(q, k, v, g, out, B, H, N, d, r, eps, None)


@pytest.mark.parametrize("f32", [False, True])
def test_forward_rejects_bad_arguments(f32):
    bad = [
        (dict(q=0), sla.INVALID_ARG),
        (dict(out=0), sla.INVALID_ARG),
        (dict(g=None), sla.INVALID_ARG),
        (dict(B=0), sla.INVALID_ARG),
        (dict(H=-1), sla.INVALID_ARG),
        (dict(N=0), sla.INVALID_ARG),
        (dict(eps=-1e-6), sla.INVALID_ARG),
        (dict(eps=float("nan")), sla.INVALID_ARG),
        (dict(eps=float("inf")), sla.INVALID_ARG),
        (dict(d=64), sla.UNSUPPORTED),
        (dict(d=256), sla.UNSUPPORTED),
        (dict(B=2, H=1 << 14, N=1 << 20), sla.UNSUPPORTED),
        (dict(k=A + STEP + 8), sla.ALIGNMENT),
        (dict(out=A + 4 * STEP + 2), sla.ALIGNMENT),
        (dict(out=A), sla.INVALID_ARG),                         # out is q
        (dict(out=A + 3 * STEP + 4096), sla.INVALID_ARG),       # out overlaps g
    ]
    for kw, want in bad:
        assert _fwd(f32=f32, **kw) == want, kw


TABLE = A + 5 * STEP          # a fake, 256-byte aligned RoPE table address


def test_forward_rejects_bad_rope_pointers():
    """The host checks only the table pointer; its contents are checked on the device."""
    assert _fwd(rope=ctypes.c_void_p(TABLE + 4)) == sla.ALIGNMENT
    assert _fwd(rope=ctypes.c_void_p(TABLE + 128)) == sla.ALIGNMENT
    assert _fwd(rope=ctypes.c_void_p(TABLE + 4), f32=True) == sla.ALIGNMENT
    # a bad table pointer never hides an earlier argument error
    assert _fwd(q=0, rope=ctypes.c_void_p(TABLE + 4)) == sla.INVALID_ARG


def test_rope_table_sizes():
    f = sla.raw_lib().sla_rope_table_floats
    # 64 header words, then N * d/2 fp16 pair words and N * d fp32 words
    assert f(22000, 128) == 64 + 22000 * 192
    assert f(159280, 128) == 64 + 159280 * 192
    assert f(4290, 256) == 64 + 4290 * 384
    assert f(1, 2) == 64 + 3
    assert f(0, 128) == 0
    assert f(10, 127) == 0
    assert f(10, 0) == 0
    assert f(1 << 30, 128) == 0                        # more words than a 32-bit offset holds
    fill = sla.raw_lib().sla_rope_table_fill
    assert fill(None, 1, 1, 1, 6, 2, 2, 2, 10000.0, None) == sla.INVALID_ARG
    assert fill(A, 1, 1, 1, 7, 3, 2, 2, 10000.0, None) == sla.INVALID_ARG     # odd band
    assert fill(A, 1, 1, 1, 8, 2, 2, 2, 10000.0, None) == sla.INVALID_ARG     # bands sum to 6
    assert fill(A, 0, 1, 1, 6, 2, 2, 2, 10000.0, None) == sla.INVALID_ARG
    assert fill(A, 1, 1, 1, 6, 2, 2, 2, 0.0, None) == sla.INVALID_ARG
    assert fill(A, 1, 1, 1, 6, 2, 2, 2, float("nan"), None) == sla.INVALID_ARG
    assert fill(A + 4, 1, 1, 1, 6, 2, 2, 2, 10000.0, None) == sla.ALIGNMENT
    assert fill(A, 1 << 12, 1 << 10, 1 << 10, 128, 44, 42, 42, 10000.0, None) == \
        sla.UNSUPPORTED
    pairs = sla.raw_lib().sla_rope_table_from_pairs
    assert pairs(None, A + STEP, 10, 128, None) == sla.INVALID_ARG
    assert pairs(A, None, 10, 128, None) == sla.INVALID_ARG
    assert pairs(A, A + STEP, 0, 128, None) == sla.INVALID_ARG
    assert pairs(A, A + STEP, 10, 127, None) == sla.INVALID_ARG
    assert pairs(A + 64, A + STEP, 10, 128, None) == sla.ALIGNMENT
    assert pairs(A, A + STEP + 4, 10, 128, None) == sla.ALIGNMENT
    assert pairs(A, A + 1024, 10, 128, None) == sla.INVALID_ARG       # pairs inside the table


def test_selftest_rejects_bad_limits_before_cuda():
    lib = sla.raw_lib()
    assert lib.sla_selftest_wait_timeout(0, None) == sla.INVALID_ARG
    assert lib.sla_selftest_wait_timeout(1000001, None) == sla.INVALID_ARG


def test_binding_rejects_mismatched_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 128)
    with pytest.raises(sla.SlaError):
        sla.linattn_forward(q, q, q, q)                      # CPU tensors
    with pytest.raises(sla.SlaError):
        sla.linattn_forward(q, q[:, :1], q, q)
    with pytest.raises(sla.SlaError):
        sla.linattn_forward(q.to(torch.float16), q, q, q)


def test_binding_rejects_bad_training_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(sla.SlaError):
        sla.linattn_forward_keep_state(q, q, q, q)           # CPU tensors
    with pytest.raises(sla.SlaError):
        sla.linattn_forward_keep_state(q, q, q, q.float())
    state = torch.zeros(sla.state_bytes(1, 2), dtype=torch.uint8)
    f = q.float()
    with pytest.raises(sla.SlaError) as err:
        sla.linattn_backward(f, f, f, f, f, state=state)     # a kept state needs bf16
    assert err.value.status in (sla.UNSUPPORTED, sla.INVALID_ARG)
    with pytest.raises(sla.SlaError):
        sla.linattn_backward(q, q, q, q, q, state=state[:100])


def test_noalloc_forward_rejects_bad_arguments_before_cuda():
    fn = sla.raw_lib().sla_linattn_forward_noalloc
    ok = dict(q=A, k=A + STEP, v=A + 2 * STEP, g=A + 3 * STEP, out=A + 4 * STEP)

    def call(status=None, **kw):
        a = dict(ok, **kw)
        return fn(a["q"], a["k"], a["v"], a["g"], a["out"], 1, 2, 256, 128, None, 1e-6,
                  status, None)

    assert call(q=0) == sla.INVALID_ARG
    assert call(out=A) == sla.INVALID_ARG
    assert call(k=A + STEP + 8) == sla.ALIGNMENT
    assert call(status=A + 6 * STEP + 2) == sla.ALIGNMENT
    assert fn(A, A + STEP, A + 2 * STEP, A + 3 * STEP, A + 4 * STEP, 1, 2, 256, 64, None, 1e-6,
              None, None) == sla.UNSUPPORTED


def test_phase_entry_points_reject_bad_arguments():
    lib = sla.raw_lib()
    st = lib.sla_linattn_state
    ap = lib.sla_linattn_apply
    K, V, S, Q, G, O = (A + i * STEP for i in range(6))
    assert lib.sla_linattn_state_bytes(2, 3, 128) == 6 * 33280
    assert lib.sla_linattn_state_bytes(2, 3, 64) == 0
    assert st(0, V, S, 1, 2, 256, 128, None, None) == sla.INVALID_ARG
    assert st(K, V, 0, 1, 2, 256, 128, None, None) == sla.INVALID_ARG
    assert st(K, V, K + 64, 1, 2, 256, 128, None, None) == sla.INVALID_ARG   # state overlaps k
    assert st(K, V, S + 8, 1, 2, 256, 128, None, None) == sla.ALIGNMENT
    assert st(K, V, S, 1, 2, 256, 96, None, None) == sla.UNSUPPORTED
    assert st(K, V, S, 0, 2, 256, 128, None, None) == sla.INVALID_ARG
    assert ap(Q, G, S, O, 1, 2, 256, 128, None, -1.0, None) == sla.INVALID_ARG
    assert ap(Q, G, S, S, 1, 2, 256, 128, None, 1e-6, None) == sla.INVALID_ARG  # out is state
    assert ap(Q, G, S, O + 4, 1, 2, 256, 128, None, 1e-6, None) == sla.ALIGNMENT
    assert ap(Q, 0, S, O, 1, 2, 256, 128, None, 1e-6, None) == sla.INVALID_ARG
    assert ap(Q, G, S, O, 1, 2, 256, 128, TABLE + 16, 1e-6, None) == sla.ALIGNMENT
    assert st(K, V, S, 1, 2, 256, 128, TABLE + 16, None) == sla.ALIGNMENT


def test_forward_cluster_rejects_bad_shapes_before_cuda():
    lib = sla.raw_lib()
    assert lib.sla_linattn_forward_cluster(0, 1, 256, 128, 0) == -1
    assert lib.sla_linattn_forward_cluster(1, 1, 0, 128, 1) == -1
    assert lib.sla_linattn_forward_cluster(1, 1, 256, 64, 0) == -1


def _bc(q=A, k=A + STEP, v=A + 2 * STEP, g=A + 3 * STEP, out=A + 4 * STEP, B=1, H=2, N=256,
        d=128, bt=64, rope=None, off=0, eps=1e-6, sin=None, sout=None):
    return sla.raw_lib().sla_linattn_forward_block_causal(q, k, v, g, out, B, H, N, d, bt, rope,
                                                          off, eps, sin, sout, None)


def test_block_causal_rejects_bad_arguments_before_cuda():
    S = A + 6 * STEP                                  # a carried-state buffer
    assert sla.carried_state_bytes(1, 2) == 2 * (128 * 128 + 128) * 4
    assert sla.carried_state_bytes(0, 2) == 0
    bad = [
        (dict(q=0), sla.INVALID_ARG),
        (dict(bt=0), sla.INVALID_ARG),
        (dict(bt=100), sla.INVALID_ARG),              # 256 tokens are not whole blocks of 100
        (dict(eps=-1.0), sla.INVALID_ARG),
        (dict(d=64), sla.UNSUPPORTED),
        (dict(off=64), sla.INVALID_ARG),              # an offset without a RoPE table
        (dict(rope=TABLE, off=-1), sla.INVALID_ARG),
        (dict(rope=TABLE + 32), sla.ALIGNMENT),
        (dict(rope=TABLE, off=0x7fffffff - 100), sla.UNSUPPORTED),   # tokens past 2^31
        (dict(sin=S + 4), sla.ALIGNMENT),
        (dict(sout=S + 8), sla.ALIGNMENT),
        (dict(sout=A + 4 * STEP + 1024), sla.INVALID_ARG),  # state out inside out
        (dict(sout=A + 1024), sla.INVALID_ARG),             # state out inside q
        (dict(sin=A + 4 * STEP), sla.INVALID_ARG),          # state in is out
        (dict(sin=S, sout=S + 1024), sla.INVALID_ARG),      # partial overlap of the states
    ]
    for kw, want in bad:
        assert _bc(**kw) == want, kw


def test_backward_rejects_bad_arguments_before_cuda():
    lib = sla.raw_lib()

    def bwd(q=A, k=A + STEP, v=A + 2 * STEP, g=A + 3 * STEP, do=A + 4 * STEP, dq=A + 5 * STEP,
            dk=A + 6 * STEP, dv=A + 7 * STEP, dg=A + 8 * STEP, N=256, d=128, eps=1e-6, f32=False):
        fn = lib.sla_linattn_backward_f32 if f32 else lib.sla_linattn_backward
        return fn(q, k, v, g, do, dq, dk, dv, dg, 1, 2, N, d, None, eps, None)

    bad = [
        (dict(do=0), sla.INVALID_ARG),
        (dict(dg=0), sla.INVALID_ARG),
        (dict(N=0), sla.INVALID_ARG),
        (dict(eps=-1.0), sla.INVALID_ARG),
        (dict(d=64), sla.UNSUPPORTED),
        (dict(dk=A + 6 * STEP + 4), sla.ALIGNMENT),
        (dict(dq=A + 2 * STEP), sla.INVALID_ARG),             # dq is v
        (dict(dv=A + 5 * STEP + 4096), sla.INVALID_ARG),      # dv overlaps dq
        (dict(dg=A + 4 * STEP + 64), sla.INVALID_ARG),        # dg overlaps dout
    ]
    for f32 in (False, True):
        for kw, want in bad:
            assert bwd(f32=f32, **kw) == want, (f32, kw)


def test_training_entries_reject_bad_arguments_before_cuda():
    lib = sla.raw_lib()
    sbytes = sla.state_bytes(1, 2)
    assert sbytes == 2 * (128 * 128 * 2 + 128 * 4)

    def keep(state=A + 5 * STEP, out=A + 4 * STEP, N=256, d=128, eps=1e-6):
        return lib.sla_linattn_forward_keep_state(A, A + STEP, A + 2 * STEP, A + 3 * STEP, out,
                                                  1, 2, N, d, None, eps, state, None)

    def bwd(state=A + 9 * STEP, dq=A + 5 * STEP, dv=A + 7 * STEP, N=256, d=128):
        return lib.sla_linattn_backward_from_state(A, A + STEP, A + 2 * STEP, A + 3 * STEP,
                                                   A + 4 * STEP, state, dq, A + 6 * STEP, dv,
                                                   A + 8 * STEP, 1, 2, N, d, None, 1e-6, None)

    for kw, want in [
        (dict(state=0), sla.INVALID_ARG),
        (dict(state=A + 5 * STEP + 8), sla.ALIGNMENT),
        (dict(state=A + 2 * STEP + 4096), sla.INVALID_ARG),      # inside v
        (dict(state=A + 4 * STEP - sbytes + 16), sla.INVALID_ARG),   # runs into out
        (dict(N=0), sla.INVALID_ARG),
        (dict(d=64), sla.UNSUPPORTED),
        (dict(eps=float("nan")), sla.INVALID_ARG),
        (dict(out=A + 4 * STEP + 2), sla.ALIGNMENT),
    ]:
        assert keep(**kw) == want, kw
    for kw, want in [
        (dict(state=0), sla.INVALID_ARG),
        (dict(state=A + 9 * STEP + 4), sla.ALIGNMENT),
        (dict(dq=A + 9 * STEP + 1024), sla.INVALID_ARG),         # dq overlaps the state
        (dict(state=A + 7 * STEP - 16), sla.INVALID_ARG),        # the state runs into dv
        (dict(N=0), sla.INVALID_ARG),
        (dict(d=64), sla.UNSUPPORTED),
    ]:
        assert bwd(**kw) == want, kw


def test_anchor_rejects_bad_arguments_before_cuda():
    lib = sla.raw_lib()
    big = 2 * 256 * 256 * 2                            # one tensor at B=1, H=2, N=256, d=256

    def anchor(q=A, k=A + 2 * STEP, v=A + 4 * STEP, g=A + 6 * STEP, out=A + 8 * STEP,
               B=1, H=2, N=256, d=256, rope=None):
        return lib.sla_anchor_forward(q, k, v, g, out, B, H, N, d, rope, None)

    assert 2 * STEP >= big
    bad = [
        (dict(q=0), sla.INVALID_ARG),
        (dict(out=0), sla.INVALID_ARG),
        (dict(N=0), sla.INVALID_ARG),
        (dict(B=-1), sla.INVALID_ARG),
        (dict(d=128), sla.UNSUPPORTED),
        (dict(B=256, H=256), sla.UNSUPPORTED),             # more than 65535 heads
        (dict(v=A + 4 * STEP + 4), sla.ALIGNMENT),
        (dict(out=A + 6 * STEP + 4096), sla.INVALID_ARG),  # out overlaps g
        (dict(rope=A + 12 * STEP + 8), sla.ALIGNMENT),     # the table is not 256-byte aligned
    ]
    for kw, want in bad:
        assert anchor(**kw) == want, kw


def test_attnres_rejects_bad_arguments_before_cuda():
    lib = sla.raw_lib()

    def agg(srcs=(A, A + STEP), M=None, T=64, C=512, w=A + 4 * STEP, eps=1e-6, out=A + 5 * STEP):
        arr = (ctypes.c_void_p * max(len(srcs), 1))(*srcs)
        return lib.sla_attnres_aggregate(arr, len(srcs) if M is None else M, T, C, w, eps, out,
                                         None)

    bad = [
        (dict(M=0), sla.INVALID_ARG),
        (dict(T=0), sla.INVALID_ARG),
        (dict(eps=-1.0), sla.INVALID_ARG),
        (dict(w=0), sla.INVALID_ARG),
        (dict(out=0), sla.INVALID_ARG),
        (dict(srcs=(A, 0)), sla.INVALID_ARG),
        (dict(srcs=tuple(A + i * STEP for i in range(9)), out=A + 12 * STEP), sla.UNSUPPORTED),
        (dict(C=300), sla.UNSUPPORTED),
        (dict(C=4352), sla.UNSUPPORTED),
        (dict(srcs=(A, A + STEP + 8)), sla.ALIGNMENT),
        (dict(w=A + 4 * STEP + 4), sla.ALIGNMENT),
        (dict(out=A + STEP + 1024), sla.INVALID_ARG),          # out overlaps a source
    ]
    for kw, want in bad:
        assert agg(**kw) == want, kw


def test_binding_rejects_bad_anchor_and_attnres_tensors():
    import torch
    q = torch.zeros(1, 2, 8, 256, dtype=torch.bfloat16)
    with pytest.raises(sla.SlaError):
        sla.anchor_forward(q, q, q, q)                       # CPU tensors
    with pytest.raises(sla.SlaError):
        sla.anchor_forward(q.float(), q, q, q)               # not bf16
    s = torch.zeros(3, 16, 512, dtype=torch.bfloat16)
    w = torch.zeros(512)
    with pytest.raises(sla.SlaError):
        sla.attnres_aggregate(s, w)                          # CPU tensors
    with pytest.raises(sla.SlaError):
        sla.attnres_aggregate(s[0], w)                       # not [M, T, C]
    with pytest.raises(sla.SlaError):
        sla.attnres_aggregate([], w)
