"""Plain fp64 CPU oracle for the forward of the gated-softmax anchor layer.

TEST INFRASTRUCTURE ONLY, like ``oracle.linattn``: nothing in the library
imports this module and it shares no code with the CUDA path.

What it computes (one (batch, head) slice; q, k, v, g are N x D):

    qr_i = R_i q_i,  kr_j = R_j k_j          3D RoPE on q and k themselves (no feature map)
    s_ij = qr_i . kr_j / sqrt(D)             scaled dot products, all N keys (no mask)
    p_ij = exp(s_ij) / sum_l exp(s_il)       softmax over the keys j
    o_i  = sigmoid(g_i) * sum_j p_ij v_j     elementwise output gate

Sources.  "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section
"Architecture"): a quarter of the layers are dense softmax anchors, with
10 heads of 256 in the 5B model and 16 heads of 256 in the 14B model, and
both kinds of layer use the Wan 3D rotary embedding.  The arXiv abstract of
2607.21553 calls them gated-softmax anchors, and the same page lists "Gated
Attention for Large Language Models" (an elementwise sigmoid gate on the
attention output) among the related work.  No page prints the formula.  The
one above is the plainest reading: standard scaled dot-product attention with
1/sqrt(D) scaling, over every token (the layer sits in a bidirectional
video DiT), and the gate g given per element, as in the linear layer.

RoPE split for D = 256: (d_t, d_h, d_w) = (88, 84, 84).  This is a reading.
The h and w bands take 2 * floor(D / 6) dimensions each and t takes the rest.
That rule gives the (44, 42, 42) printed for D = 128, and the pages give no
other split.  The rotation itself is ``oracle.linattn.rope_rotate`` with the
angles of ``oracle.linattn.rope3d_angles``.

Every function works in float64 on numpy arrays.  The softmax subtracts the
row maximum before exponentiating, which leaves each p_ij unchanged.
"""
from __future__ import annotations

import numpy as np

from .linattn import RopeSpec, _as64, rope3d_angles, rope_rotate, sigmoid

__all__ = [
    "anchor_split",
    "anchor_head",
    "anchor_forward",
    "anchor_forward_rows",
]


def anchor_split(D):
    """(d_t, d_h, d_w) for head dim D: h and w take 2 * floor(D / 6) each, t the rest."""
    hw = 2 * (D // 6)
    return D - 2 * hw, hw, hw


def _rotate(x, angles):
    return x if angles is None else rope_rotate(x, angles)


def _scores(qr, kr):
    """s = qr kr^T / sqrt(D)."""
    return qr @ kr.T / np.sqrt(qr.shape[1])


def _softmax(s):
    """Row-wise softmax over the last axis."""
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _gate(g, y):
    return sigmoid(g) * y


def anchor_head(q, k, v, g, angles=None, q_angles=None):
    """Output [Nq, D] of one head.  angles: [Nk, D/2] for the keys (and for the
    queries too, unless q_angles gives the queries' own rows), or None."""
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    qa = angles if q_angles is None else q_angles
    qr = _rotate(q, qa)
    kr = _rotate(k, angles)
    return _gate(g, _softmax(_scores(qr, kr)) @ v)


def _resolve(rope, N, D):
    if rope is None:
        return None
    if isinstance(rope, RopeSpec):
        if rope.n_tokens != N or rope.d != D:
            raise ValueError("RoPE grid/split does not match the tensor shape")
        return rope3d_angles(rope)
    angles = np.asarray(rope, dtype=np.float64)
    if angles.shape != (N, D // 2):
        raise ValueError("angle table must be [N, D/2]")
    return angles


def anchor_forward(q, k, v, g, rope=None):
    """[B, H, N, D] forward in float64.  rope: a RopeSpec, an [N, D/2] angle array, or None."""
    q, k, v, g = (_as64(x) for x in (q, k, v, g))
    B, H, N, D = q.shape
    angles = _resolve(rope, N, D)
    out = np.empty((B, H, N, D))
    for b in range(B):
        for h in range(H):
            out[b, h] = anchor_head(q[b, h], k[b, h], v[b, h], g[b, h], angles)
    return out


def anchor_forward_rows(q, k, v, g, rows, rope=None, heads=None):
    """Outputs at selected query rows only: {(b, h): [len(rows), D]}, each row
    still attending to all N keys."""
    rows = np.asarray(rows, dtype=np.int64)
    B, H, N, D = q.shape
    angles = _resolve(rope, N, D)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    result = {}
    for b, h in heads:
        qq, gg = _as64(q[b, h][rows]), _as64(g[b, h][rows])
        kk, vv = _as64(k[b, h]), _as64(v[b, h])
        qa = None if angles is None else angles[rows]
        result[(b, h)] = anchor_head(qq, kk, vv, gg, angles, q_angles=qa)
    return result
