"""Block-causal form with a carried state, CUDA path vs the fp64 oracle, through
the C ABI (sla_linattn_forward_block_causal).

The carried state is compared as well as the outputs.  Small shapes are
compared element by element; they cover several block sizes, including blocks
that end inside a 64- or 128-token tile, one block per head, and one token
per block.  Chained calls, an incoming state, in-place update and a RoPE
offset are covered.  The 720p shape in blocks of five frames is compared on
sampled rows.  The bound is max|err| / max|ref| <= 1e-2 for the bf16 outputs.
The carried state is summed in fp32, so z and, without RoPE, S (phi(k) of a bf16
key is exact in bf16) meet 1e-4.  With RoPE the tensor cores take the rotated
keys rounded to bf16 (2^-9 relative per term), so S meets the bf16 bound.
"""
import numpy as np
import pytest
import torch

import oracle.block_causal as bc
import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL, STATE_TOL = 1e-2, 1e-4


def _s_tol(rope):
    return TOL if rope else STATE_TOL


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _np64(t):
    return t.detach().float().cpu().double().numpy()


def _rel(out, ref):
    return float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))


def _state_np(state, B, H):
    S, z = _sla().carried_state_parts(state)
    return S.detach().cpu().double().numpy(), z.detach().cpu().double().numpy()


def _state_t(S, z, device):
    B, H = z.shape[:2]
    flat = np.concatenate([S.reshape(B, H, -1), z], axis=2)
    return torch.tensor(flat, dtype=torch.float32, device=device).contiguous()


def _run(tensors, block_tokens, device, rope=None, offset=0, state_in=None, eps=1e-6):
    q, k, v, g = (t.to(device) for t in tensors)
    out, st = _sla().linattn_forward_block_causal(q, k, v, g, block_tokens, rope=rope,
                                                  rope_offset=offset, eps=eps, state_in=state_in)
    assert _sla().last_device_status(device=device) == 0
    return out, st


CASES = [
    # (B, H, grid, block_frames, rope)
    (1, 2, (4, 2, 16), 1, True),      # blocks of 32 tokens, inside one tile
    (2, 3, (3, 7, 11), 1, False),     # 77-token blocks, ragged in both tile sizes
    (1, 2, (6, 8, 16), 2, True),      # 256-token blocks
    (1, 3, (6, 10, 13), 3, True),     # 390-token blocks
    (2, 2, (3, 10, 10), 3, False),    # one block per head
    (1, 1, (4, 5, 30), 1, True),      # 150-token blocks
]


@pytest.mark.parametrize("B,H,grid,frames,rope", CASES,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-bt{f*g[1]*g[2]}-{'rope' if r else 'norope'}"
                              for b, h, g, f, r in CASES])
def test_block_causal_elementwise(B, H, grid, frames, rope, cuda_device):
    sla = _sla()
    wl = Workload("bc", B=B, H=H, grid=grid, rope=rope, block_frames=frames)
    tensors = make_inputs(wl, seed=21)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device) if rope else None
    out, st = _run(tensors, wl.block_tokens, cuda_device, rope=table)
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if rope else None
    ref, (S, z) = bc.linattn_forward_block_causal(*tensors, wl.block_tokens, 1e-6, spec)
    assert _rel(_np64(out), ref) <= TOL
    S_gpu, z_gpu = _state_np(st, B, H)
    assert _rel(S_gpu, S) <= _s_tol(rope) and _rel(z_gpu, z) <= STATE_TOL


def test_token_blocks_are_causal_attention(cuda_device):
    """One token per block: causal linear attention (RoPE on)."""
    sla = _sla()
    wl = Workload("tok", B=1, H=2, grid=(70, 1, 1), rope=True, split=(44, 42, 42), block_frames=1)
    tensors = make_inputs(wl, seed=22)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    out, _ = _run(tensors, 1, cuda_device, rope=table)
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base)
    ref, _ = bc.linattn_forward_block_causal(*tensors, 1, 1e-6, spec)
    assert _rel(_np64(out), ref) <= TOL


def test_chained_calls_and_incoming_state(cuda_device):
    """Three calls over consecutive stretches, each starting from the previous
    state and its RoPE offset; the last one updates its state in place."""
    sla = _sla()
    wl = Workload("chain", B=2, H=2, grid=(6, 6, 9), rope=True, block_frames=1)
    tensors = make_inputs(wl, seed=23)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    bt = wl.block_tokens
    cuts = [0, 2 * bt, 3 * bt, 6 * bt]
    outs, state = [], None
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = tuple(t[:, :, a:b].contiguous() for t in tensors)
        q, k, v, g = (t.to(cuda_device) for t in part)
        if state is None:
            o, state = sla.linattn_forward_block_causal(q, k, v, g, bt, rope=table, rope_offset=a)
        else:
            o, state = sla.linattn_forward_block_causal(q, k, v, g, bt, rope=table, rope_offset=a,
                                                        state_in=state, state_out=state)
        outs.append(o)
    assert sla.last_device_status(device=cuda_device) == 0
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base)
    ref, (S, z) = bc.linattn_forward_block_causal(*tensors, bt, 1e-6, spec)
    assert _rel(_np64(torch.cat(outs, dim=2)), ref) <= TOL
    S_gpu, z_gpu = _state_np(state, 2, 2)
    assert _rel(S_gpu, S) <= _s_tol(True) and _rel(z_gpu, z) <= STATE_TOL


def test_given_incoming_state(cuda_device):
    sla = _sla()
    wl = Workload("sin", B=1, H=2, grid=(4, 4, 8), rope=False, block_frames=2)
    tensors = make_inputs(wl, seed=24)
    rng = np.random.default_rng(5)
    S0 = rng.standard_normal((1, 2, 128, 128)) * 3.0
    z0 = rng.uniform(0.0, 40.0, (1, 2, 128))        # a sum of ReLU features is >= 0
    st_in = _state_t(S0, z0, cuda_device)
    out, st = _run(tensors, wl.block_tokens, cuda_device, state_in=st_in)
    ref, (S, z) = bc.linattn_forward_block_causal(*tensors, wl.block_tokens, 1e-6, None, 0, (S0, z0))
    assert _rel(_np64(out), ref) <= TOL
    S_gpu, z_gpu = _state_np(st, 1, 2)
    assert _rel(S_gpu, S) <= STATE_TOL and _rel(z_gpu, z) <= STATE_TOL


def test_one_block_matches_the_bidirectional_forward(cuda_device):
    sla = _sla()
    wl = Workload("one", B=2, H=2, grid=(3, 11, 13), rope=True)
    tensors = make_inputs(wl, seed=25)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    out, _ = _run(tensors, wl.N, cuda_device, rope=table)
    q, k, v, g = (t.to(cuda_device) for t in tensors)
    fwd = sla.linattn_forward(q, k, v, g, rope=table)
    ref = ol.linattn_forward(*tensors, eps=1e-6, rope=ol.RopeSpec(*wl.grid, *wl.split))
    assert _rel(_np64(out), ref) <= TOL
    assert _rel(_np64(out), _np64(fwd)) <= TOL


def test_720p_blocks_of_five_frames_sampled_rows(cuda_device):
    sla = _sla()
    wl = WORKLOADS["5b_720p_block5"]
    tensors = make_inputs(wl, seed=0)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    out, st = _run(tensors, wl.block_tokens, cuda_device, rope=table)
    rows = sample_rows(wl.N, 40)
    heads = [(0, 0), (0, 11), (1, 19)]
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base)
    ref = bc.linattn_block_causal_rows(*tensors, wl.block_tokens, rows, 1e-6, spec, heads=heads)
    got = np.stack([_np64(out[b, h][rows]) for b, h in heads])
    want = np.stack([ref[bh] for bh in heads])
    assert _rel(got, want) <= wl.tol
    # the final state of one head against the oracle's sum over all tokens
    q, k, v, g = tensors
    S, z = ol.linattn_state(k[1, 19].double().numpy(), v[1, 19].double().numpy(),
                            ol.rope3d_angles(spec))
    S_gpu, z_gpu = _state_np(st, wl.B, wl.H)
    assert _rel(S_gpu[1, 19], S) <= _s_tol(True) and _rel(z_gpu[1, 19], z) <= STATE_TOL
