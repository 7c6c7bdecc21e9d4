"""Plain fp64 CPU oracle for the gated bidirectional linear-attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA path.

What it computes (one (batch, head) slice; q, k, v, g are N x d):

    phi(x)      = max(x, 0)                                   feature map
    kr_j        = R_j phi(k_j)   (R_j = identity without RoPE)
    S           = sum_j kr_j v_j^T            (d x d)         state
    z           = sum_j phi(k_j)              (d)             normaliser (unrotated)
    qr_i        = R_i phi(q_i)
    num_i       = qr_i^T S                    (d)
    den_i       = phi(q_i) . z + eps          (scalar, unrotated q)
    o_i         = sigmoid(g_i) * num_i / den_i                elementwise gate

Sources.  "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section
"Architecture") names the layer: gated, bidirectional (the sums run over every
token j, no causal mask) linear attention with Wan 3D rotary position
embeddings.  The article "SANA-Video 2.0: Hybrid Attention for Faster
High-Resolution Video Generation" (Key points, first bullet) and the arXiv
abstract of 2607.21553 call it the gated linear attention used for most token
mixing.  The pages print no formula; the one above (ReLU feature map, output
gate sigmoid(g), eps in the denominator, RoPE on the numerator only) is the
plainest reading that the rest of the pages support, and every reading is
listed in the design notes.

3D RoPE reading ("Wan 3D rotary position embeddings", same section of the
NVlabs page; RoFormer is among the cited prior work).  The head dimension d is
split into three even bands (d_t, d_h, d_w) = (44, 42, 42) for d = 128, in the
order t, h, w.  Band a rotates its adjacent pairs (x_{2p}, x_{2p+1}) as the
complex number x_{2p} + i x_{2p+1} multiplied by exp(i * pos_a * theta_{a,j}),
where j is the pair index inside the band and theta_{a,j} = base^(-2j/d_a).
Token n of a T x Hs x Ws latent grid sits at (t, h, w) with
n = (t * Hs + h) * Ws + w ("(1, 1, 1) latent patches" on the NVlabs page).

Every function works in float64 on numpy arrays.  No blocking, fusion or
reordering is done beyond the definition: the two contractions are plain
matrix products.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "feature_map",
    "sigmoid",
    "RopeSpec",
    "rope3d_positions",
    "rope3d_thetas",
    "rope3d_angles",
    "rope_rotate",
    "linattn_state",
    "linattn_apply",
    "linattn_head",
    "linattn_forward",
    "linattn_forward_rows",
]


def feature_map(x):
    """phi(x) = max(x, 0), the ReLU feature map applied to q and k."""
    return np.maximum(np.asarray(x, dtype=np.float64), 0.0)


def sigmoid(g):
    """The output gate 1 / (1 + exp(-g)), in float64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


class RopeSpec:
    """A T x Hs x Ws latent grid with head-dim split (d_t, d_h, d_w) and base."""

    def __init__(self, T, Hs, Ws, dt=44, dh=42, dw=42, base=10000.0):
        for name, val in (("dt", dt), ("dh", dh), ("dw", dw)):
            if val < 0 or val % 2:
                raise ValueError(f"RoPE band {name}={val} must be even and >= 0")
        self.T, self.Hs, self.Ws = int(T), int(Hs), int(Ws)
        self.dt, self.dh, self.dw = int(dt), int(dh), int(dw)
        self.base = float(base)

    @property
    def n_tokens(self):
        return self.T * self.Hs * self.Ws

    @property
    def d(self):
        return self.dt + self.dh + self.dw


def rope3d_positions(spec: RopeSpec):
    """(t, h, w) of every token, row-major over the grid: n = (t*Hs + h)*Ws + w."""
    n = np.arange(spec.n_tokens, dtype=np.int64)
    w = n % spec.Ws
    h = (n // spec.Ws) % spec.Hs
    t = n // (spec.Ws * spec.Hs)
    return t, h, w


def rope3d_thetas(width, base):
    """Frequency ladder of one band of even width: theta_j = base^(-2j/width)."""
    j = np.arange(width // 2, dtype=np.float64)
    return base ** (-2.0 * j / width)


def rope3d_angles(spec: RopeSpec):
    """Angle of every (token, pair): an [N, d/2] float64 array.

    Pairs [0, d_t/2) take the t coordinate, the next d_h/2 pairs take h and the
    last d_w/2 pairs take w, each band with its own frequency ladder.
    """
    t, h, w = rope3d_positions(spec)
    bands = []
    for pos, width in ((t, spec.dt), (h, spec.dh), (w, spec.dw)):
        bands.append(np.outer(pos.astype(np.float64), rope3d_thetas(width, spec.base)))
    return np.concatenate(bands, axis=1)


def rope_rotate(x, angles):
    """Rotate adjacent pairs (x_{2p}, x_{2p+1}) of each row by angles[:, p].

    x: [N, d] float64, angles: [N, d/2].  Returns a new array; the pair is
    treated as the complex number x_{2p} + i x_{2p+1} times exp(i angle).
    """
    x = np.asarray(x, dtype=np.float64)
    c = np.cos(angles)
    s = np.sin(angles)
    x0 = x[:, 0::2]
    x1 = x[:, 1::2]
    out = np.empty_like(x)
    out[:, 0::2] = x0 * c - x1 * s
    out[:, 1::2] = x0 * s + x1 * c
    return out


def linattn_state(k, v, angles=None):
    """State of one head: S = sum_j R_j phi(k_j) v_j^T and z = sum_j phi(k_j).

    k, v: [N, d].  angles: [N, d/2] or None (no RoPE).  S is rotated when RoPE
    is on; z never is (the denominator uses the unrotated features).
    """
    kp = feature_map(k)
    kr = kp if angles is None else rope_rotate(kp, angles)
    v = np.asarray(v, dtype=np.float64)
    S = kr.T @ v
    z = kp.sum(axis=0)
    return S, z


def linattn_apply(q, g, S, z, eps, angles=None):
    """Outputs o_i = sigmoid(g_i) * (R_i phi(q_i))^T S / (phi(q_i) . z + eps).

    q, g: [M, d] rows to evaluate; angles: [M, d/2] for those rows or None.
    """
    qp = feature_map(q)
    qr = qp if angles is None else rope_rotate(qp, angles)
    num = qr @ S
    den = qp @ z + eps
    return sigmoid(g) * num / den[:, None]


def linattn_head(q, k, v, g, eps, angles=None):
    """Full forward of one (batch, head) slice: [N, d] inputs to [N, d] output."""
    S, z = linattn_state(k, v, angles)
    return linattn_apply(q, g, S, z, eps, angles)


def _as64(x):
    if hasattr(x, "detach"):  # a torch tensor: exact upcast of its values
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def linattn_forward(q, k, v, g, eps=1e-6, rope=None):
    """[B, H, N, d] forward in float64.  rope: a RopeSpec, an [N, d/2] angle array, or None."""
    q, k, v, g = (_as64(x) for x in (q, k, v, g))
    B, H, N, d = q.shape
    angles = _resolve_angles(rope, N, d)
    out = np.empty((B, H, N, d), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            out[b, h] = linattn_head(q[b, h], k[b, h], v[b, h], g[b, h], eps, angles)
    return out


def linattn_forward_rows(q, k, v, g, rows, eps=1e-6, rope=None, heads=None):
    """Outputs at selected token rows only, each head's state over all N tokens.

    rows: 1-D integer array of token indices (shared by all heads).
    heads: iterable of (b, h) pairs, default all.  Returns {(b, h): [len(rows), d]}.
    """
    rows = np.asarray(rows, dtype=np.int64)
    B, H, N, d = q.shape
    angles = _resolve_angles(rope, N, d)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    result = {}
    for b, h in heads:
        kk, vv = _as64(k[b, h]), _as64(v[b, h])
        S, z = linattn_state(kk, vv, angles)
        qq, gg = _as64(q[b, h][rows]), _as64(g[b, h][rows])
        ang = None if angles is None else angles[rows]
        result[(b, h)] = linattn_apply(qq, gg, S, z, eps, ang)
    return result


def _resolve_angles(rope, N, d):
    if rope is None:
        return None
    if isinstance(rope, RopeSpec):
        if rope.n_tokens != N or rope.d != d:
            raise ValueError("RoPE grid/split does not match the tensor shape")
        return rope3d_angles(rope)
    angles = np.asarray(rope, dtype=np.float64)
    if angles.shape != (N, d // 2):
        raise ValueError("angle table must be [N, d/2]")
    return angles
