"""Gated-softmax anchor forward, CUDA path vs the fp64 oracle
(oracle/softmax_anchor.py), through the C ABI (sla_anchor_forward).

Small shapes are compared element by element over several 128-query and
64-key tiles with ragged tails, RoPE on and off.  The full-size workloads are
compared on sampled query rows (each row still attends to every key).  The
bound is max|err| / max|ref| <= 1e-2 (bf16 inputs and output, fp32
accumulation, softmax weights rounded to bf16 for the second product).
"""
import numpy as np
import pytest
import torch

import oracle.linattn as ol
import oracle.softmax_anchor as oa
from gated_linear_attention_attn_b300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL = 1e-2


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _np64(t):
    return t.detach().float().cpu().double().numpy()


def _rel(out, ref):
    return float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))


def _wl(B, H, grid, rope):
    return Workload("anchor", B=B, H=H, grid=grid, d=256, rope=rope, split=(88, 84, 84),
                    layer="anchor")


def _spec(wl):
    return ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None


def _run(wl, tensors, device):
    sla = _sla()
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=device) if wl.rope else None
    out = sla.anchor_forward(*(t.to(device) for t in tensors), rope=rope)
    assert sla.last_device_status(device=device) == 0
    return out


CASES = [
    (1, 1, (1, 1, 1), False),        # one token
    (1, 1, (1, 1, 7), False),
    (1, 2, (1, 8, 16), True),        # 128: one whole query tile, two key tiles
    (2, 1, (1, 1, 129), False),      # a one-row query tail, a one-key tail
    (1, 2, (3, 10, 10), True),       # 300
    (2, 3, (2, 9, 17), True),        # 306, six heads
    (1, 1, (1, 1, 1000), False),
    (1, 2, (4, 16, 20), True),       # 1280: ten query tiles
]


@pytest.mark.parametrize("B,H,grid,rope", CASES,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-{'rope' if r else 'norope'}"
                              for b, h, g, r in CASES])
def test_anchor_elementwise(B, H, grid, rope, cuda_device):
    wl = _wl(B, H, grid, rope)
    tensors = make_inputs(wl, seed=17)
    got = _run(wl, tensors, cuda_device)
    want = oa.anchor_forward(*tensors, rope=_spec(wl))
    assert _rel(_np64(got), want) <= TOL


def test_anchor_peaked_scores(cuda_device):
    """Large scores (q and k scaled by 6: score std about 36) exercise the
    running-maximum rescale of the accumulator many times per row.  No RoPE:
    rotated rows rounded to bf16 would move such scores by about 0.1."""
    wl = _wl(1, 2, (2, 10, 30), False)
    q, k, v, g = make_inputs(wl, seed=5)
    q, k = (x.float().mul(6.0).to(torch.bfloat16) for x in (q, k))
    got = _run(wl, (q, k, v, g), cuda_device)
    want = oa.anchor_forward(q, k, v, g, rope=_spec(wl))
    assert _rel(_np64(got), want) <= TOL


def test_anchor_increasing_scores(cuda_device):
    """Scores that grow along the keys (the maximum moves in every key tile)."""
    wl = _wl(1, 1, (1, 1, 900), False)
    q, k, v, g = make_inputs(wl, seed=6)
    q = torch.ones_like(q) * 0.5
    ramp = torch.linspace(0.0, 3.0, wl.N).view(1, 1, -1, 1)
    k = (ramp * torch.ones(1, 1, wl.N, wl.d)).to(torch.bfloat16)
    got = _run(wl, (q, k, v, g), cuda_device)
    want = oa.anchor_forward(q, k, v, g)
    assert _rel(_np64(got), want) <= TOL


@pytest.mark.parametrize("name", ["anchor_5b_480p", "anchor_14b_480p", "anchor_5b_720p"])
def test_anchor_full_size_sampled_rows(name, cuda_device):
    wl = WORKLOADS[name]
    tensors = make_inputs(wl, seed=0)
    got = _run(wl, tensors, cuda_device)
    rows = sample_rows(wl.N, 24)
    heads = [(0, 0), (wl.B - 1, wl.H - 1)]
    ref = oa.anchor_forward_rows(*tensors, rows, rope=_spec(wl), heads=heads)
    g_gpu = np.stack([_np64(got[b, h][rows]) for b, h in heads])
    g_ref = np.stack([ref[bh] for bh in heads])
    assert _rel(g_gpu, g_ref) <= wl.tol
    assert torch.isfinite(got.float()).all()
