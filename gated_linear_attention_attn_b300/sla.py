"""Python binding of libsla.so: the gated bidirectional linear-attention forward.

This module only marshals arguments: it turns torch CUDA tensors into device
pointers, sizes and the current stream, and calls the C ABI declared in
``include/sla.h``.  Every step of the computation runs in the library's CUDA
kernels.  Importing it fails loudly if the library has not been built
(``python -m gated_linear_attention_attn_b300.build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m gated_linear_attention_attn_b300.build`"
        " (the forward has no other implementation)")

_lib = ctypes.CDLL(LIB_PATH)

OK, INVALID_ARG, UNSUPPORTED, ALIGNMENT, CUDA_ERROR, DEVICE_TIMEOUT = range(6)
HEAD_DIM = 128


_vp, _int, _flt = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_lib.sla_rope_table_floats.argtypes = [_int] * 2
_lib.sla_rope_table_floats.restype = ctypes.c_size_t
_lib.sla_rope_table_fill.argtypes = [_vp] + [_int] * 7 + [_flt, _vp]
_lib.sla_rope_table_fill.restype = _int
_lib.sla_rope_table_from_pairs.argtypes = [_vp, _vp, _int, _int, _vp]
_lib.sla_rope_table_from_pairs.restype = _int
_FWD_ARGS = [_vp] * 5 + [_int] * 4 + [_vp, _flt, _vp]
for _name in ("sla_linattn_forward", "sla_linattn_forward_f32"):
    getattr(_lib, _name).argtypes = _FWD_ARGS
    getattr(_lib, _name).restype = _int
_lib.sla_linattn_state_bytes.argtypes = [_int] * 3
_lib.sla_linattn_state_bytes.restype = ctypes.c_size_t
_lib.sla_linattn_state.argtypes = [_vp] * 3 + [_int] * 4 + [_vp, _vp]
_lib.sla_linattn_state.restype = _int
_lib.sla_linattn_apply.argtypes = [_vp] * 4 + [_int] * 4 + [_vp, _flt, _vp]
_lib.sla_linattn_apply.restype = _int
_lib.sla_linattn_forward_noalloc.argtypes = _FWD_ARGS[:-1] + [_vp, _vp]
_lib.sla_linattn_forward_noalloc.restype = _int
_lib.sla_linattn_carried_state_bytes.argtypes = [_int] * 3
_lib.sla_linattn_carried_state_bytes.restype = ctypes.c_size_t
_lib.sla_linattn_forward_block_causal.argtypes = ([_vp] * 5 + [_int] * 5 +
                                                  [_vp, _int, _flt, _vp, _vp, _vp])
_lib.sla_linattn_forward_block_causal.restype = _int
_BWD_ARGS = [_vp] * 9 + [_int] * 4 + [_vp, _flt, _vp]
for _name in ("sla_linattn_backward", "sla_linattn_backward_f32"):
    getattr(_lib, _name).argtypes = _BWD_ARGS
    getattr(_lib, _name).restype = _int
_lib.sla_linattn_forward_keep_state.argtypes = _FWD_ARGS[:-1] + [_vp, _vp]
_lib.sla_linattn_forward_keep_state.restype = _int
_lib.sla_linattn_backward_from_state.argtypes = [_vp] * 10 + [_int] * 4 + [_vp, _flt, _vp]
_lib.sla_linattn_backward_from_state.restype = _int
_lib.sla_anchor_forward.argtypes = [_vp] * 5 + [_int] * 4 + [_vp, _vp]
_lib.sla_anchor_forward.restype = _int
_lib.sla_attnres_aggregate.argtypes = [ctypes.POINTER(_vp), _int, _int, _int, _vp, _flt, _vp,
                                       _vp]
_lib.sla_attnres_aggregate.restype = _int
_lib.sla_linattn_forward_cluster.argtypes = [_int] * 5
_lib.sla_linattn_forward_cluster.restype = _int
_lib.sla_status_string.argtypes = [_int]
_lib.sla_status_string.restype = ctypes.c_char_p
_lib.sla_last_device_status.argtypes = [_vp]
_lib.sla_last_device_status.restype = _int
_lib.sla_selftest_wait_timeout.argtypes = [ctypes.c_uint, _vp]
_lib.sla_selftest_wait_timeout.restype = _int

EXPORTED = ("sla_rope_table_floats", "sla_rope_table_fill", "sla_rope_table_from_pairs",
            "sla_linattn_forward",
            "sla_linattn_forward_f32", "sla_linattn_state_bytes", "sla_linattn_state",
            "sla_linattn_apply", "sla_linattn_forward_noalloc", "sla_linattn_forward_cluster",
            "sla_linattn_carried_state_bytes", "sla_linattn_forward_block_causal",
            "sla_linattn_backward", "sla_linattn_backward_f32",
            "sla_linattn_forward_keep_state", "sla_linattn_backward_from_state",
            "sla_anchor_forward",
            "sla_attnres_aggregate", "sla_status_string", "sla_last_device_status",
            "sla_selftest_wait_timeout")


class SlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def status_string(status: int) -> str:
    return _lib.sla_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise SlaError(status, where)


def _stream_handle(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


class RopeTable:
    """A RoPE table on one device (``sla_rope_table_fill``): a header, then every
    token's d/2 (cos, sin) pairs as fp16 and as fp32 (layout in ``include/sla.h``).

    ``RopeTable(grid, split, base)`` builds the 3D table of a latent grid;
    ``RopeTable.from_pairs(pairs)`` wraps caller-given fp32 pairs [N, d/2, 2].
    """

    def __init__(self, grid: Sequence[int], split: Sequence[int] = (44, 42, 42),
                 base: float = 10000.0, device="cuda", stream=None):
        T, Hs, Ws = (int(x) for x in grid)
        dt, dh, dw = (int(x) for x in split)
        d = dt + dh + dw
        self.device = torch.device(device)
        self.grid, self.split, self.base, self.d = (T, Hs, Ws), (dt, dh, dw), float(base), d
        self.n_tokens = T * Hs * Ws
        self.table = self._alloc(self.n_tokens, d)
        with torch.cuda.device(self.device):
            _check(_lib.sla_rope_table_fill(self.table.data_ptr(), T, Hs, Ws, d, dt, dh, dw,
                                            self.base, _stream_handle(stream, self.device)),
                   "sla_rope_table_fill")

    def _alloc(self, n: int, d: int) -> torch.Tensor:
        words = int(_lib.sla_rope_table_floats(n, d))
        if words == 0:
            raise SlaError(INVALID_ARG, "sla_rope_table_floats")
        return torch.empty(words, dtype=torch.float32, device=self.device)

    @classmethod
    def from_pairs(cls, pairs: torch.Tensor, stream=None) -> "RopeTable":
        """A table from an fp32 CUDA tensor [N, d/2, 2] of (cos, sin) per token and pair
        (``sla_rope_table_from_pairs``)."""
        if pairs.dtype != torch.float32 or pairs.dim() != 3 or pairs.shape[2] != 2 \
                or pairs.device.type != "cuda" or not pairs.is_contiguous():
            raise SlaError(INVALID_ARG, "from_pairs: pairs must be a contiguous fp32 "
                                        "[N, d/2, 2] CUDA tensor")
        self = cls.__new__(cls)
        self.device = pairs.device
        self.grid, self.split, self.base = None, None, None
        self.n_tokens, self.d = int(pairs.shape[0]), 2 * int(pairs.shape[1])
        self.table = self._alloc(self.n_tokens, self.d)
        with torch.cuda.device(self.device):
            _check(_lib.sla_rope_table_from_pairs(self.table.data_ptr(), pairs.data_ptr(),
                                                  self.n_tokens, self.d,
                                                  _stream_handle(stream, self.device)),
                   "sla_rope_table_from_pairs")
        return self

    @property
    def ptr(self) -> int:
        """The table's device address: the ``rope_table`` argument of the C ABI."""
        return self.table.data_ptr()

    def header(self):
        """The header words as a list of ints (tag, version, N, d, T, Hs, Ws, dt, dh, dw,
        base bits, offset of the fp16 rows, offset of the fp32 pairs)."""
        return self.table[:13].view(torch.int32).cpu().tolist()

    def token_rows(self):
        """The fp16 part as an [N, d/2, 2] float16 tensor of (cos, sin)."""
        p = self.d // 2
        off = 64
        return self.table[off:off + self.n_tokens * p].view(torch.float16).view(
            self.n_tokens, p, 2)

    def pairs(self):
        """The fp32 part as an [N, d/2, 2] float32 tensor of (cos, sin)."""
        p = self.d // 2
        off = 64 + self.n_tokens * p
        return self.table[off:off + 2 * self.n_tokens * p].view(self.n_tokens, p, 2)


def _rope_ptr(rope: Optional[RopeTable]):
    return rope.ptr if rope is not None else None


def linattn_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                    out: Optional[torch.Tensor] = None, rope: Optional[RopeTable] = None,
                    eps: float = 1e-6, stream: Optional[torch.cuda.Stream] = None
                    ) -> torch.Tensor:
    """o = sigmoid(g) * (R phi(q)) S / (phi(q) . z + eps) for [B, H, N, d] CUDA tensors.

    bf16 tensors go to ``sla_linattn_forward``, fp32 tensors to
    ``sla_linattn_forward_f32``.  Asynchronous on ``stream`` (default: the
    current stream).  Raises SlaError with the library's status on bad input.
    """
    if q.dim() != 4:
        raise SlaError(INVALID_ARG, "linattn_forward: q must be [B, H, N, d]")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device:
            raise SlaError(INVALID_ARG, f"linattn_forward: {name} differs from q")
        if not t.is_contiguous():
            raise SlaError(INVALID_ARG, f"linattn_forward: {name} is not contiguous")
    if q.device.type != "cuda":
        raise SlaError(INVALID_ARG, "linattn_forward: tensors must be on a CUDA device")
    if q.dtype == torch.bfloat16:
        fn = _lib.sla_linattn_forward
    elif q.dtype == torch.float32:
        fn = _lib.sla_linattn_forward_f32
    else:
        raise SlaError(UNSUPPORTED, f"linattn_forward: dtype {q.dtype}")
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() \
            or out.device != q.device:
        raise SlaError(INVALID_ARG, "linattn_forward: out must match q")
    B, H, N, d = q.shape
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(q.device):
        _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), out.data_ptr(),
                  B, H, N, d, rope_c, float(eps), _stream_handle(stream, q.device)),
               fn.__name__)
    return out


ANCHOR_HEAD_DIM = 256
ANCHOR_SPLIT = (88, 84, 84)


def anchor_forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                   out: Optional[torch.Tensor] = None, rope: Optional[RopeTable] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """o = sigmoid(g) * softmax((R q)(R k)^T / sqrt(d)) v for [B, H, N, 256] bf16 CUDA tensors
    (``sla_anchor_forward``).  Asynchronous on ``stream`` (default: the current stream)."""
    _check_bf16("q", q)
    for name, t in (("k", k), ("v", v), ("g", g)):
        _check_bf16(name, t, like=q)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_bf16("out", out, like=q)
    B, H, N, d = q.shape
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(q.device):
        _check(_lib.sla_anchor_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                                       out.data_ptr(), B, H, N, d, rope_c,
                                       _stream_handle(stream, q.device)),
               "sla_anchor_forward")
    return out


def attnres_aggregate(sources, w: torch.Tensor, eps: float = 1e-6,
                      out: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """x(t) = sum_n softmax_n(w . rmsnorm(s_n(t))) s_n(t) (``sla_attnres_aggregate``).

    sources: a list of M bf16 [T, C] CUDA tensors, or one [M, T, C] tensor; w: fp32 [C].
    """
    if isinstance(sources, torch.Tensor):
        if sources.dim() != 3:
            raise SlaError(INVALID_ARG, "attnres_aggregate: a sources tensor must be [M, T, C]")
        sources = list(sources.unbind(0))
    if not sources:
        raise SlaError(INVALID_ARG, "attnres_aggregate: no sources")
    first = sources[0]
    for t in sources:
        if t.dtype != torch.bfloat16 or t.dim() != 2 or t.shape != first.shape \
                or t.device != first.device or t.device.type != "cuda" or not t.is_contiguous():
            raise SlaError(INVALID_ARG, "attnres_aggregate: sources must be contiguous bf16 "
                                        "[T, C] CUDA tensors of one shape")
    T, C = first.shape
    if w.dtype != torch.float32 or w.shape != (C,) or w.device != first.device \
            or not w.is_contiguous():
        raise SlaError(INVALID_ARG, "attnres_aggregate: w must be a contiguous fp32 [C] tensor")
    if out is None:
        out = torch.empty_like(first)
    elif out.shape != first.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() \
            or out.device != first.device:
        raise SlaError(INVALID_ARG, "attnres_aggregate: out must be a bf16 [T, C] tensor")
    ptrs = (_vp * len(sources))(*[t.data_ptr() for t in sources])
    with torch.cuda.device(first.device):
        _check(_lib.sla_attnres_aggregate(ptrs, len(sources), T, C, w.data_ptr(), float(eps),
                                          out.data_ptr(), _stream_handle(stream, first.device)),
               "sla_attnres_aggregate")
    return out


def _check_bf16(name, t, like=None):
    if t.dtype != torch.bfloat16 or t.dim() != 4 or t.device.type != "cuda" \
            or not t.is_contiguous():
        raise SlaError(INVALID_ARG, f"{name} must be a contiguous [B, H, N, d] bf16 CUDA tensor")
    if like is not None and (t.shape != like.shape or t.device != like.device):
        raise SlaError(INVALID_ARG, f"{name} differs from its partner tensor")


def state_bytes(B: int, H: int, d: int = HEAD_DIM) -> int:
    """Bytes of the per-head state that ``linattn_state`` writes."""
    return int(_lib.sla_linattn_state_bytes(B, H, d))


def linattn_state(k: torch.Tensor, v: torch.Tensor, rope: Optional[RopeTable] = None,
                  state: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Phase 1 (bf16): the heads' S and z from k and v, as a uint8 device buffer."""
    _check_bf16("k", k)
    _check_bf16("v", v, like=k)
    B, H, N, d = k.shape
    nbytes = state_bytes(B, H, d)
    if nbytes == 0:
        raise SlaError(UNSUPPORTED, "linattn_state: shape")
    if state is None:
        state = torch.empty(nbytes, dtype=torch.uint8, device=k.device)
    elif state.numel() * state.element_size() < nbytes or not state.is_contiguous():
        raise SlaError(INVALID_ARG, "linattn_state: state buffer too small")
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(k.device):
        _check(_lib.sla_linattn_state(k.data_ptr(), v.data_ptr(), state.data_ptr(), B, H, N, d,
                                      rope_c, _stream_handle(stream, k.device)),
               "sla_linattn_state")
    return state


def linattn_apply(q: torch.Tensor, g: torch.Tensor, state: torch.Tensor,
                  out: Optional[torch.Tensor] = None, rope: Optional[RopeTable] = None,
                  eps: float = 1e-6, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Phase 2 (bf16): o from q, g and a state written by ``linattn_state``."""
    _check_bf16("q", q)
    _check_bf16("g", g, like=q)
    B, H, N, d = q.shape
    if state.device != q.device or not state.is_contiguous() \
            or state.numel() * state.element_size() < state_bytes(B, H, d):
        raise SlaError(INVALID_ARG, "linattn_apply: state does not match q")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_bf16("out", out, like=q)
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(q.device):
        _check(_lib.sla_linattn_apply(q.data_ptr(), g.data_ptr(), state.data_ptr(),
                                      out.data_ptr(), B, H, N, d, rope_c, float(eps),
                                      _stream_handle(stream, q.device)),
               "sla_linattn_apply")
    return out


def linattn_forward_keep_state(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               g: torch.Tensor, out: Optional[torch.Tensor] = None,
                               rope: Optional[RopeTable] = None, eps: float = 1e-6,
                               state: Optional[torch.Tensor] = None,
                               stream: Optional[torch.cuda.Stream] = None):
    """The bf16 forward that also writes the heads' states for the backward
    (``sla_linattn_forward_keep_state``): returns (out, state), state a uint8 device
    buffer of ``state_bytes(B, H)`` bytes as ``linattn_state`` writes it."""
    _check_bf16("q", q)
    for name, t in (("k", k), ("v", v), ("g", g)):
        _check_bf16(name, t, like=q)
    B, H, N, d = q.shape
    nbytes = state_bytes(B, H, d)
    if nbytes == 0:
        raise SlaError(UNSUPPORTED, "linattn_forward_keep_state: shape")
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_bf16("out", out, like=q)
    if state is None:
        state = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    elif state.device != q.device or not state.is_contiguous() \
            or state.numel() * state.element_size() < nbytes:
        raise SlaError(INVALID_ARG, "linattn_forward_keep_state: state buffer too small")
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(q.device):
        _check(_lib.sla_linattn_forward_keep_state(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), out.data_ptr(), B, H, N, d,
            rope_c, float(eps), state.data_ptr(), _stream_handle(stream, q.device)),
            "sla_linattn_forward_keep_state")
    return out, state


def last_device_status(stream: Optional[torch.cuda.Stream] = None, device="cuda") -> int:
    """Synchronise the stream and read (and clear) the device status word."""
    dev = torch.device(device)
    with torch.cuda.device(dev):
        return _lib.sla_last_device_status(_stream_handle(stream, dev))


def selftest_wait_timeout(limit_us: int = 1000, stream: Optional[torch.cuda.Stream] = None,
                          device="cuda") -> None:
    """Launch the bounded-wait self-test (``sla_selftest_wait_timeout``): one thread waits
    on an mbarrier nobody arrives at and gives up after ``limit_us`` microseconds."""
    dev = torch.device(device)
    with torch.cuda.device(dev):
        _check(_lib.sla_selftest_wait_timeout(int(limit_us), _stream_handle(stream, dev)),
               "sla_selftest_wait_timeout")


def linattn_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                     dout: torch.Tensor, rope: Optional[RopeTable] = None, eps: float = 1e-6,
                     grads: Optional[Sequence[torch.Tensor]] = None,
                     stream: Optional[torch.cuda.Stream] = None,
                     state: Optional[torch.Tensor] = None):
    """(dq, dk, dv, dg) of sum(dout * o) for [B, H, N, d] CUDA tensors (bf16 or fp32;
    ``sla_linattn_backward`` / ``sla_linattn_backward_f32``).  grads: four output
    tensors to fill, else new ones.  state (bf16 only): the heads' states of the
    forward (``linattn_forward_keep_state`` or ``linattn_state``), used instead of
    recomputing them (``sla_linattn_backward_from_state``)."""
    for name, t in (("k", k), ("v", v), ("g", g), ("dout", dout)):
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device \
                or not t.is_contiguous():
            raise SlaError(INVALID_ARG, f"linattn_backward: {name} differs from q")
    if q.dim() != 4 or not q.is_contiguous() or q.device.type != "cuda":
        raise SlaError(INVALID_ARG, "linattn_backward: q must be a contiguous [B, H, N, d] "
                                    "CUDA tensor")
    if state is not None:
        if q.dtype != torch.bfloat16:
            raise SlaError(UNSUPPORTED, "linattn_backward: a given state needs bf16 tensors")
        if state.device != q.device or not state.is_contiguous() \
                or state.numel() * state.element_size() < state_bytes(*q.shape[:2], q.shape[3]):
            raise SlaError(INVALID_ARG, "linattn_backward: state does not match q")
        fn = _lib.sla_linattn_backward_from_state
    elif q.dtype == torch.bfloat16:
        fn = _lib.sla_linattn_backward
    elif q.dtype == torch.float32:
        fn = _lib.sla_linattn_backward_f32
    else:
        raise SlaError(UNSUPPORTED, f"linattn_backward: dtype {q.dtype}")
    if grads is None:
        grads = tuple(torch.empty_like(q) for _ in range(4))
    for t in grads:
        if t.shape != q.shape or t.dtype != q.dtype or t.device != q.device \
                or not t.is_contiguous():
            raise SlaError(INVALID_ARG, "linattn_backward: gradient tensors must match q")
    B, H, N, d = q.shape
    rope_c = _rope_ptr(rope)
    ins = [q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), dout.data_ptr()]
    if state is not None:
        ins.append(state.data_ptr())
    with torch.cuda.device(q.device):
        _check(fn(*ins, *(t.data_ptr() for t in grads), B, H, N, d, rope_c, float(eps),
                  _stream_handle(stream, q.device)), fn.__name__)
    return tuple(grads)


CARRIED_FLOATS = HEAD_DIM * HEAD_DIM + HEAD_DIM


def carried_state_bytes(B: int, H: int, d: int = HEAD_DIM) -> int:
    """Bytes of a carried (S, z) state for B*H heads (``sla_linattn_carried_state_bytes``)."""
    return int(_lib.sla_linattn_carried_state_bytes(B, H, d))


def carried_state_parts(state: torch.Tensor):
    """Views (S [B, H, 128, 128], z [B, H, 128]) of a [B, H, 128*128 + 128] carried state."""
    B, H = state.shape[:2]
    S = state[..., :HEAD_DIM * HEAD_DIM].view(B, H, HEAD_DIM, HEAD_DIM)
    return S, state[..., HEAD_DIM * HEAD_DIM:]


def linattn_forward_block_causal(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                 g: torch.Tensor, block_tokens: int,
                                 out: Optional[torch.Tensor] = None,
                                 rope: Optional[RopeTable] = None, rope_offset: int = 0,
                                 eps: float = 1e-6, state_in: Optional[torch.Tensor] = None,
                                 state_out=True, stream: Optional[torch.cuda.Stream] = None):
    """Block-causal forward with a carried state (bf16; ``sla_linattn_forward_block_causal``).

    state_in: None or a float32 [B, H, 128*128 + 128] tensor (S row-major,
    then z).  state_out: True to allocate one, a tensor to fill (may be
    state_in), or None for none.  Returns (out, state_out).
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        _check_bf16(name, t, like=q if name != "q" else None)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check_bf16("out", out, like=q)
    if state_out is True:
        state_out = torch.empty(B, H, CARRIED_FLOATS, dtype=torch.float32, device=q.device)
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None and (t.dtype != torch.float32 or t.device != q.device
                              or not t.is_contiguous() or t.numel() != B * H * CARRIED_FLOATS):
            raise SlaError(INVALID_ARG, f"{name} must be a contiguous float32 [B, H, "
                                        f"{CARRIED_FLOATS}] tensor on q's device")
    rope_c = _rope_ptr(rope)
    with torch.cuda.device(q.device):
        _check(_lib.sla_linattn_forward_block_causal(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), out.data_ptr(),
            B, H, N, d, int(block_tokens), rope_c, int(rope_offset), float(eps),
            state_in.data_ptr() if state_in is not None else None,
            state_out.data_ptr() if state_out is not None else None,
            _stream_handle(stream, q.device)), "sla_linattn_forward_block_causal")
    return out, state_out


def forward_cluster(B: int, H: int, N: int, rope: bool, d: int = HEAD_DIM,
                    device=None) -> int:
    """Cluster size of the fused one-launch forward for this shape, 0 for the
    state and apply launches (``sla_linattn_forward_cluster``)."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    with torch.cuda.device(dev):
        c = int(_lib.sla_linattn_forward_cluster(B, H, N, d, 1 if rope else 0))
    if c < 0:
        raise SlaError(INVALID_ARG, "sla_linattn_forward_cluster")
    return c


class forward_kernel:
    """Context manager that sets SLA_FORWARD_KERNEL ("fused", "split" or
    "auto") for the calls made inside it."""

    def __init__(self, path: str):
        if path not in ("fused", "split", "auto"):
            raise ValueError(f"forward kernel {path!r}: expected fused, split or auto")
        self.path = path

    def __enter__(self):
        self._old = os.environ.get("SLA_FORWARD_KERNEL")
        os.environ["SLA_FORWARD_KERNEL"] = self.path
        return self

    def __exit__(self, *exc):
        if self._old is None:
            os.environ.pop("SLA_FORWARD_KERNEL", None)
        else:
            os.environ["SLA_FORWARD_KERNEL"] = self._old
        return False


def launches_per_forward(dtype: torch.dtype, B: int = 1, H: int = 1, N: int = 1,
                         rope: bool = False, device=None) -> int:
    """Kernels one forward call launches: the fused kernel alone, or the state
    reduction and the apply (the fp32 path: the state and apply kernels)."""
    if dtype == torch.bfloat16 and forward_cluster(B, H, N, rope, device=device) > 0:
        return 1
    return 2


def raw_lib() -> ctypes.CDLL:
    """The loaded library, for callers that pass raw pointers."""
    return _lib


class LinAttnFunction(torch.autograd.Function):
    """The layer as a torch autograd function, for training: the forward keeps each
    head's state (bf16: ``linattn_forward_keep_state``) and the backward reuses it
    (``linattn_backward(..., state=...)``); fp32 tensors take the fp32 forward and the
    recomputing fp32 backward.  Only argument marshalling happens here; every step runs
    in the library.  Use ``linattn(q, k, v, g, rope, eps)``."""

    @staticmethod
    def forward(ctx, q, k, v, g, rope, eps):
        q, k, v, g = (t.contiguous() for t in (q, k, v, g))
        if q.dtype == torch.bfloat16:
            out, state = linattn_forward_keep_state(q, k, v, g, rope=rope, eps=eps)
        else:
            out, state = linattn_forward(q, k, v, g, rope=rope, eps=eps), None
        ctx.save_for_backward(q, k, v, g)
        ctx.state, ctx.rope, ctx.eps = state, rope, eps
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, g = ctx.saved_tensors
        grads = linattn_backward(q, k, v, g, dout.contiguous(), rope=ctx.rope, eps=ctx.eps,
                                 state=ctx.state)
        ctx.state = None
        return (*grads, None, None)


def linattn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
            rope: Optional[RopeTable] = None, eps: float = 1e-6) -> torch.Tensor:
    """The layer's forward with autograd support (see ``LinAttnFunction``)."""
    return LinAttnFunction.apply(q, k, v, g, rope, eps)
