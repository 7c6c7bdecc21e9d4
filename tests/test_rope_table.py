"""The device RoPE table: its values against the oracle's float64 angles, its header, the
table made from caller-given pairs, and tables that do not fit a call, which every kernel
that rotates must refuse on the device (status word -> SLA_ERR_INVALID_ARG) without
reading past the header."""
import numpy as np
import pytest
import torch

import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


@pytest.mark.parametrize("grid,split", [((25, 22, 40), (44, 42, 42)),
                                        ((181, 22, 40), (44, 42, 42)),
                                        ((3, 5, 7), (8, 6, 114)),
                                        ((2, 1, 1), (128, 0, 0)),
                                        ((3, 4, 5), (88, 84, 84))])
def test_table_matches_oracle_angles(grid, split, cuda_device):
    sla = _sla()
    rt = sla.RopeTable(grid, split, 10000.0, device=cuda_device)
    spec = ol.RopeSpec(*grid, *split, base=10000.0)
    ang = ol.rope3d_angles(spec)                              # [N, d/2] float64
    cs = rt.pairs().double().cpu().numpy()                    # [N, d/2, 2]
    assert cs.shape == ang.shape + (2,)
    assert np.max(np.abs(cs[..., 0] - np.cos(ang))) <= 1e-6
    assert np.max(np.abs(cs[..., 1] - np.sin(ang))) <= 1e-6
    # the fp16 rows: every pair of every token, the fp32 value rounded to fp16
    tok = rt.token_rows()
    assert torch.equal(tok, rt.pairs().to(torch.float16))
    tok = tok.double().cpu().numpy()
    assert np.max(np.abs(tok[..., 0] - np.cos(ang))) <= 2.5e-4
    assert np.max(np.abs(tok[..., 1] - np.sin(ang))) <= 2.5e-4


def test_table_header(cuda_device):
    sla = _sla()
    rt = sla.RopeTable((25, 22, 40), (44, 42, 42), 10000.0, device=cuda_device)
    h = rt.header()
    base_bits = int(np.array([10000.0], dtype=np.float32).view(np.int32)[0])
    assert h == [0x33414c53, 1, 22000, 128, 25, 22, 40, 44, 42, 42, base_bits, 64,
                 64 + 22000 * 64]
    assert rt.table.numel() == 64 + 22000 * 192
    assert torch.all(rt.table[13:64].view(torch.int32) == 0)


def test_table_from_pairs_equals_fill(cuda_device):
    """A table made from the filled table's fp32 pairs holds the same rows and gives the
    same forward output, bit for bit; its header records no grid."""
    sla = _sla()
    wl = Workload("rp", B=1, H=3, grid=(3, 10, 12), rope=True)
    filled = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    pairs = filled.pairs().clone()
    made = sla.RopeTable.from_pairs(pairs)
    del pairs                                                # the copy does not keep it
    torch.cuda.synchronize(cuda_device)
    assert torch.equal(made.table[64:], filled.table[64:])
    assert made.header()[:4] == [0x33414c53, 1, wl.N, 128]
    assert made.header()[4:11] == [0] * 7
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=5))
    for path in ("fused", "split"):
        with sla.forward_kernel(path):
            a = sla.linattn_forward(q, k, v, g, rope=filled)
            b = sla.linattn_forward(q, k, v, g, rope=made)
        assert sla.last_device_status(device=cuda_device) == sla.OK
        assert torch.equal(a, b)


def _bad_tables(sla, device, n, d):
    """Tables a call over n tokens of head dim d must refuse."""
    grid_more = sla.RopeTable((1, 1, n + 1), (d - 4, 2, 2), device=device)      # n + 1 tokens
    grid_less = sla.RopeTable((1, 1, max(n - 1, 1)), (d - 4, 2, 2), device=device)
    other_d = sla.RopeTable((1, 1, n), (2 * d - 4, 2, 2), device=device)          # 2d
    zeros = sla.RopeTable((1, 1, n), (d - 4, 2, 2), device=device)
    zeros.table.zero_()                                                           # no header
    bad = [grid_more, other_d, zeros]
    if n > 1:
        bad.append(grid_less)
    return bad


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("path", ["fused", "split"])
def test_forward_refuses_tables_that_do_not_fit(dtype, path, cuda_device):
    sla = _sla()
    wl = Workload("badrope", B=1, H=2, grid=(2, 8, 16), dtype=dtype, rope=True)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=6))
    good = sla.RopeTable(wl.grid, wl.split, device=cuda_device)
    assert sla.last_device_status(device=cuda_device) == sla.OK
    with sla.forward_kernel(path):
        for table in _bad_tables(sla, cuda_device, wl.N, 128):
            sla.linattn_forward(q, k, v, g, rope=table)
            assert sla.last_device_status(device=cuda_device) == sla.INVALID_ARG
            assert sla.last_device_status(device=cuda_device) == sla.OK     # read and cleared
        out = sla.linattn_forward(q, k, v, g, rope=good)
    assert sla.last_device_status(device=cuda_device) == sla.OK
    ref = ol.linattn_forward(*make_inputs(wl, seed=6), eps=wl.eps,
                             rope=ol.RopeSpec(*wl.grid, *wl.split, base=wl.base))
    got = out.float().cpu().double().numpy()
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= wl.tol


def test_other_entry_points_refuse_tables_that_do_not_fit(cuda_device):
    sla = _sla()
    wl = Workload("badrope2", B=1, H=2, grid=(2, 8, 16), rope=True)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=7))
    short = sla.RopeTable((1, 8, 16), wl.split, device=cuda_device)     # half the tokens
    calls = [
        lambda: sla.linattn_state(k, v, rope=short),
        lambda: sla.linattn_backward(q, k, v, g, q, rope=short),
        lambda: sla.linattn_backward(q.float(), k.float(), v.float(), g.float(), q.float(),
                                     rope=short),
        # the second half of the sequence: tokens 128..255 of a 128-token table
        lambda: sla.linattn_forward_block_causal(q[:, :, :128].contiguous(),
                                                 k[:, :, :128].contiguous(),
                                                 v[:, :, :128].contiguous(),
                                                 g[:, :, :128].contiguous(), 64, rope=short,
                                                 rope_offset=128),
    ]
    state = sla.linattn_state(k, v)
    calls.append(lambda: sla.linattn_apply(q, g, state, rope=short))
    aw = Workload("badrope_anchor", B=1, H=2, grid=(2, 8, 16), d=256, rope=True,
                  split=(88, 84, 84), layer="anchor")
    aq, ak, av, ag = (t.to(cuda_device) for t in make_inputs(aw, seed=8))
    d128 = sla.RopeTable(aw.grid, (44, 42, 42), device=cuda_device)    # built for d = 128
    calls.append(lambda: sla.anchor_forward(aq, ak, av, ag, rope=d128))
    assert sla.last_device_status(device=cuda_device) == sla.OK
    for i, call in enumerate(calls):
        call()
        assert sla.last_device_status(device=cuda_device) == sla.INVALID_ARG, i
    # a block-causal stretch inside the table is fine
    sla.linattn_forward_block_causal(q[:, :, :128].contiguous(), k[:, :, :128].contiguous(),
                                     v[:, :, :128].contiguous(), g[:, :, :128].contiguous(), 64,
                                     rope=sla.RopeTable(wl.grid, wl.split, device=cuda_device),
                                     rope_offset=128)
    assert sla.last_device_status(device=cuda_device) == sla.OK
