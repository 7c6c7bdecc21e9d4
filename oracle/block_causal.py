"""Plain fp64 CPU oracle for the block-causal form with a carried state.

TEST INFRASTRUCTURE ONLY, like ``oracle.linattn``: nothing in the library
imports this module and it shares no code with the CUDA path.

Source.  The SANA-Video model card (page "SANA-Video_2B_720p", "SANA-Video
Model Card", second key innovation, "Constant-Memory KV Cache for Block Linear
Attention"; model type "Block Linear Diffusion Transformer") describes a
block-wise autoregressive form. It relies on the cumulative property of
linear attention: global context is kept at a fixed memory cost, instead of
in a growing KV cache.  The page gives no formula; the reading built here is:

* the N tokens of a head form consecutive blocks of ``block_tokens`` tokens
  (whole latent frames, so each block is a contiguous range of the t-outermost
  token order);
* a token in block b attends to every token of blocks 0..b: its own block in
  both directions (the block's frames are generated together), the earlier
  blocks through the carried state;
* the carried state of a head is the pair (S, z) of the bidirectional layer
  summed over all tokens seen so far, plus an optional incoming state
  (S0, z0) from earlier calls.  So for token i of block b:

      S_b = S0 + sum_{j in blocks 0..b} R_j phi(k_j) v_j^T
      z_b = z0 + sum_{j in blocks 0..b} phi(k_j)
      o_i = sigmoid(g_i) * (R_i phi(q_i))^T S_b / (phi(q_i) . z_b + eps)

  and the outgoing state is (S_{last}, z_{last}).  With block_tokens = N and
  no incoming state this is the bidirectional layer; with block_tokens = 1 it
  is the causal linear attention.

RoPE positions are absolute: a call that covers tokens [n0, n0 + N) of a
latent grid rotates them with the grid's angles of those tokens, so chained
calls on consecutive blocks give the same result as one call on all of them.
"""
from __future__ import annotations

import numpy as np

from .linattn import RopeSpec, _as64, linattn_apply, linattn_state, rope3d_angles

__all__ = [
    "block_angles",
    "linattn_block_causal_head",
    "linattn_forward_block_causal",
    "linattn_block_causal_rows",
]


def block_angles(rope, N, d, rope_offset=0):
    """Angles [N, d/2] of tokens [rope_offset, rope_offset + N) of a grid, or None."""
    if rope is None:
        return None
    if isinstance(rope, RopeSpec):
        if rope.d != d or rope_offset < 0 or rope_offset + N > rope.n_tokens:
            raise ValueError("RoPE grid/split does not cover the tokens of this call")
        return rope3d_angles(rope)[rope_offset:rope_offset + N]
    angles = np.asarray(rope, dtype=np.float64)
    if angles.shape != (N, d // 2):
        raise ValueError("angle table must be [N, d/2]")
    return angles


def _check_blocks(N, block_tokens):
    if block_tokens < 1 or N % block_tokens:
        raise ValueError("N must be a whole number of blocks")
    return N // block_tokens


def linattn_block_causal_head(q, k, v, g, block_tokens, eps, angles=None, S0=None, z0=None):
    """One (batch, head) slice.  Returns (o [N, d], S [d, d], z [d]).

    Blocks are taken in order; each block's keys and values are added to the
    running state before the block's queries read it.
    """
    q, k, v, g = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g))
    N, d = q.shape
    nb = _check_blocks(N, block_tokens)
    S = np.zeros((d, d)) if S0 is None else np.array(S0, dtype=np.float64)
    z = np.zeros(d) if z0 is None else np.array(z0, dtype=np.float64)
    out = np.empty((N, d))
    for b in range(nb):
        sl = slice(b * block_tokens, (b + 1) * block_tokens)
        ang = None if angles is None else angles[sl]
        Sb, zb = linattn_state(k[sl], v[sl], ang)
        S = S + Sb
        z = z + zb
        out[sl] = linattn_apply(q[sl], g[sl], S, z, eps, ang)
    return out, S, z


def linattn_forward_block_causal(q, k, v, g, block_tokens, eps=1e-6, rope=None, rope_offset=0,
                                 state_in=None):
    """[B, H, N, d] block-causal forward in float64.

    rope: a RopeSpec of the whole grid (the call covers its tokens
    [rope_offset, rope_offset + N)), an [N, d/2] angle array, or None.
    state_in: None or a pair (S0 [B, H, d, d], z0 [B, H, d]).
    Returns (out [B, H, N, d], (S [B, H, d, d], z [B, H, d])).
    """
    q, k, v, g = (_as64(x) for x in (q, k, v, g))
    B, H, N, d = q.shape
    angles = block_angles(rope, N, d, rope_offset)
    out = np.empty((B, H, N, d))
    S_out = np.empty((B, H, d, d))
    z_out = np.empty((B, H, d))
    for b in range(B):
        for h in range(H):
            S0 = None if state_in is None else state_in[0][b, h]
            z0 = None if state_in is None else state_in[1][b, h]
            out[b, h], S_out[b, h], z_out[b, h] = linattn_block_causal_head(
                q[b, h], k[b, h], v[b, h], g[b, h], block_tokens, eps, angles, S0, z0)
    return out, (S_out, z_out)


def linattn_block_causal_rows(q, k, v, g, block_tokens, rows, eps=1e-6, rope=None,
                              rope_offset=0, heads=None):
    """Outputs at selected token rows only ({(b, h): [len(rows), d]}), each
    row read against the running state of its block."""
    rows = np.asarray(rows, dtype=np.int64)
    B, H, N, d = q.shape
    nb = _check_blocks(N, block_tokens)
    angles = block_angles(rope, N, d, rope_offset)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    result = {}
    for b, h in heads:
        kk, vv = _as64(k[b, h]), _as64(v[b, h])
        S = np.zeros((d, d))
        z = np.zeros(d)
        states = []
        for blk in range(nb):
            sl = slice(blk * block_tokens, (blk + 1) * block_tokens)
            Sb, zb = linattn_state(kk[sl], vv[sl], None if angles is None else angles[sl])
            S = S + Sb
            z = z + zb
            states.append((S, z))
        qq, gg = _as64(q[b, h][rows]), _as64(g[b, h][rows])
        out = np.empty((len(rows), d))
        for r, i in enumerate(rows):
            Sb, zb = states[int(i) // block_tokens]
            ang = None if angles is None else angles[i:i + 1]
            out[r] = linattn_apply(qq[r:r + 1], gg[r:r + 1], Sb, zb, eps, ang)[0]
        result[(b, h)] = out
    return result
