"""Plain fp64 CPU oracle for the backward of the gated linear-attention layer.

TEST INFRASTRUCTURE ONLY, like ``oracle.linattn``: nothing in the library
imports this module and it shares no code with the CUDA path.

Source.  "SANA-Video 2.0" (NVlabs/Sana docs/sana_video2.md, section
"Training") trains the models of the section "Architecture" (from scratch, or
from a checkpoint), so the layer's backward is part of the method.  The
pages give no formula for it.  This module states the gradient of
L = sum(dO * o) for the forward of ``oracle.linattn`` (one head, q, k, v, g
and dO are N x d), by the chain rule:

    a_i    = dO_i * sigmoid(g_i) / den_i            dL/dnum_i
    dg_i   = dO_i * num_i / den_i * s_i (1 - s_i)   with s_i = sigmoid(g_i)
    dden_i = -(a_i . num_i) / den_i                 dL/dden_i
    dS     = sum_i qr_i a_i^T                       d x d
    dz     = sum_i dden_i phi(q_i)                  d
    dq_i   = [q_i > 0] * (R_i^T (S a_i) + dden_i z)
    dk_j   = [k_j > 0] * (R_j^T (dS v_j) + dz)
    dv_j   = dS^T kr_j

where num_i = qr_i^T S, den_i = phi(q_i) . z + eps, qr_i = R_i phi(q_i) and
kr_j = R_j phi(k_j).  The ReLU derivative at 0 is taken as 0.
"""
from __future__ import annotations

import numpy as np

from .linattn import _as64, _resolve_angles, feature_map, rope_rotate, sigmoid

__all__ = ["linattn_head_backward", "linattn_backward", "linattn_backward_rows"]


def _rot(x, angles, sign=1.0):
    return x if angles is None else rope_rotate(x, sign * angles)


def _head_state(k, v, angles):
    kp = feature_map(k)
    kr = _rot(kp, angles)
    return kp, kr, kr.T @ np.asarray(v, dtype=np.float64), kp.sum(axis=0)


def _query_terms(q, g, do, S, z, eps, angles):
    """(qp, qr, a, dg, dden) of a block of query rows."""
    qp = feature_map(q)
    qr = _rot(qp, angles)
    num = qr @ S
    den = qp @ z + eps
    s = sigmoid(g)
    do = np.asarray(do, dtype=np.float64)
    a = do * s / den[:, None]
    dg = do * num / den[:, None] * s * (1.0 - s)
    dden = -(a * num).sum(axis=1) / den
    return qp, qr, a, dg, dden


def linattn_head_backward(q, k, v, g, do, eps, angles=None):
    """(dq, dk, dv, dg) of one head, each N x d."""
    q, k, v, g, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, do))
    kp, kr, S, z = _head_state(k, v, angles)
    qp, qr, a, dg, dden = _query_terms(q, g, do, S, z, eps, angles)
    dS = qr.T @ a
    dz = qp.T @ dden
    dq = (q > 0) * (_rot(a @ S.T, angles, -1.0) + dden[:, None] * z[None, :])
    dk = (k > 0) * (_rot(v @ dS.T, angles, -1.0) + dz[None, :])
    dv = kr @ dS
    return dq, dk, dv, dg


def linattn_backward(q, k, v, g, do, eps=1e-6, rope=None):
    """[B, H, N, d] backward in float64; returns (dq, dk, dv, dg)."""
    q, k, v, g, do = (_as64(x) for x in (q, k, v, g, do))
    B, H, N, d = q.shape
    angles = _resolve_angles(rope, N, d)
    outs = [np.empty((B, H, N, d)) for _ in range(4)]
    for b in range(B):
        for h in range(H):
            res = linattn_head_backward(q[b, h], k[b, h], v[b, h], g[b, h], do[b, h], eps, angles)
            for o, r in zip(outs, res):
                o[b, h] = r
    return tuple(outs)


def linattn_backward_rows(q, k, v, g, do, rows, eps=1e-6, rope=None, heads=None):
    """The four gradients at selected token rows only: {(b, h): (dq, dk, dv, dg)}, each
    [len(rows), d].  The head's S, z, dS and dz are still summed over all N tokens."""
    rows = np.asarray(rows, dtype=np.int64)
    B, H, N, d = q.shape
    angles = _resolve_angles(rope, N, d)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    result = {}
    for b, h in heads:
        qq, kk, vv, gg, dd = (_as64(x[b, h]) for x in (q, k, v, g, do))
        kp, kr, S, z = _head_state(kk, vv, angles)
        qp, qr, a, dg, dden = _query_terms(qq, gg, dd, S, z, eps, angles)
        dS = qr.T @ a
        dz = qp.T @ dden
        ang = None if angles is None else angles[rows]
        dq = (qq[rows] > 0) * (_rot(a[rows] @ S.T, ang, -1.0) + dden[rows, None] * z[None, :])
        dk = (kk[rows] > 0) * (_rot(vv[rows] @ dS.T, ang, -1.0) + dz[None, :])
        dv = kr[rows] @ dS
        result[(b, h)] = (dq, dk, dv, dg[rows])
    return result
