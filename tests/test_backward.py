"""Backward of the layer, CUDA path vs the fp64 backward oracle, through the C
ABI (sla_linattn_backward, sla_linattn_backward_f32).

Small shapes are compared element by element, for all four gradients and
several tiles with a ragged tail, RoPE on and off.  The 480p workloads are
compared on sampled token rows.  The bound is max|err| / max|ref| per
gradient: 1e-5 for fp32 inputs, 1e-2 for bf16 inputs (fp32 arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle.backward as ob
import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}
NAMES = ("dq", "dk", "dv", "dg")


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _np64(t):
    return t.detach().float().cpu().double().numpy()


def _rel(out, ref):
    return float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))


def _inputs(wl, seed):
    q, k, v, g = make_inputs(wl, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1000)
    dout = torch.randn(q.shape, generator=gen).to(wl.dtype)
    return q, k, v, g, dout


def _run(wl, tensors, device):
    sla = _sla()
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=device) if wl.rope else None
    grads = sla.linattn_backward(*(t.to(device) for t in tensors), rope=rope, eps=wl.eps)
    assert sla.last_device_status(device=device) == 0
    return grads


CASES = [
    (1, 1, (1, 1, 7), torch.bfloat16, False),
    (1, 2, (1, 8, 16), torch.bfloat16, True),
    (2, 3, (1, 1, 129), torch.bfloat16, False),
    (1, 2, (3, 10, 10), torch.bfloat16, True),
    (2, 4, (2, 9, 17), torch.bfloat16, True),
    (3, 1, (1, 1, 1000), torch.bfloat16, False),
    # 240 query tiles: more than one per CTA, with heads changing inside a CTA
    (2, 40, (1, 4, 75), torch.bfloat16, True),
    (1, 2, (4, 8, 8), torch.float32, True),
    (2, 1, (1, 1, 300), torch.float32, False),
]


@pytest.mark.parametrize("B,H,grid,dtype,rope", CASES,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-{str(dt)[6:]}-{'rope' if r else 'norope'}"
                              for b, h, g, dt, r in CASES])
def test_backward_elementwise(B, H, grid, dtype, rope, cuda_device):
    wl = Workload("bwd", B=B, H=H, grid=grid, dtype=dtype, rope=rope)
    tensors = _inputs(wl, seed=41)
    got = _run(wl, tensors, cuda_device)
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if rope else None
    want = ob.linattn_backward(*tensors, eps=wl.eps, rope=spec)
    for name, a, b in zip(NAMES, got, want):
        assert _rel(_np64(a), b) <= TOL[dtype], name


@pytest.mark.parametrize("name", ["5b_480p", "14b_480p", "5b_720p"])
def test_backward_full_size_sampled_rows(name, cuda_device):
    wl = WORKLOADS[name]
    tensors = _inputs(wl, seed=0)
    got = _run(wl, tensors, cuda_device)
    rows = sample_rows(wl.N, 24)
    heads = [(0, 0), (1, wl.H - 1)]
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
    ref = ob.linattn_backward_rows(*tensors, rows, wl.eps, spec, heads)
    for i, gname in enumerate(NAMES):
        g_gpu = np.stack([_np64(got[i][b, h][rows]) for b, h in heads])
        g_ref = np.stack([ref[bh][i] for bh in heads])
        assert _rel(g_gpu, g_ref) <= wl.tol, gname


def test_zero_upstream_gradient_gives_zero_gradients(cuda_device):
    wl = Workload("zero", B=1, H=2, grid=(2, 5, 20), rope=True)
    q, k, v, g, dout = _inputs(wl, seed=42)
    got = _run(wl, (q, k, v, g, torch.zeros_like(dout)), cuda_device)
    for name, t in zip(NAMES, got):
        assert torch.count_nonzero(t) == 0, name
