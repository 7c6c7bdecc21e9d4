"""The allocation-free forward (sla_linattn_forward_noalloc) against sla_linattn_forward.

Some callers cannot let a library allocate device memory: a framework whose caching
allocator already holds the GPU's memory, a runtime whose enqueue path forbids
allocation, or a latency-critical loop that cannot afford the device-wide
synchronisation of cudaMalloc/cudaFree.  For them the library runs the same kernels with
their scratch in a fixed array of its device code.  This file checks, through the C ABI,
that two calls in a row give what the ordinary entry point gives, and that a shape whose
scratch would not fit is refused before anything runs.  It is collected last so that a
run stopping at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from gated_linear_attention_attn_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2   # max|err| / max|ref| for bf16 inputs, as in the parity tests


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _args(q, k, v, g, out, rope):
    B, H, N, d = q.shape
    r = rope.ptr if rope is not None else None
    return [q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), out.data_ptr(), B, H, N, d,
            r, 1e-6]


@pytest.mark.parametrize("path", ["auto", "split"])
@pytest.mark.parametrize("wl,seeds", [
    (Workload("na_rope", B=2, H=3, grid=(4, 11, 13), rope=True), (11, 12)),
    (Workload("na_norope", B=1, H=4, grid=(1, 1, 300), rope=False), (13, 14)),
    (Workload("na_multi", B=2, H=4, grid=(4, 10, 110), rope=True), (16, 17)),
])
def test_noalloc_matches_forward_on_two_calls(wl, seeds, path, cuda_device, monkeypatch):
    """Both launch plans: the fused one needs no scratch, the two launches use the array.
    The two entry points run the same kernels and sum the partial states in the same
    order, so their outputs agree bit for bit; the first call is also held to the oracle.
    The last shape spreads every head over many CTAs, whose shared merge counts through
    the array."""
    monkeypatch.setenv("SLA_FORWARD_KERNEL", path)
    sla = _sla()
    lib = sla.raw_lib()
    stream = torch.cuda.current_stream(cuda_device)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device) if wl.rope else None
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for seed in seeds:                    # two calls in a row, different inputs
        q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=seed))
        ref = torch.empty_like(q)
        got = torch.full_like(q, float("nan"))
        with torch.cuda.device(cuda_device):
            rc = lib.sla_linattn_forward(*_args(q, k, v, g, ref, rope), stream.cuda_stream)
            assert rc == sla.OK, sla.status_string(rc)
            rc = lib.sla_linattn_forward_noalloc(*_args(q, k, v, g, got, rope),
                                                 status.data_ptr(), stream.cuda_stream)
            assert rc == sla.OK, sla.status_string(rc)
        torch.cuda.synchronize(cuda_device)
        assert int(status.item()) == 0
        assert torch.equal(got, ref)
        if seed == seeds[0]:
            import oracle.linattn as ol
            spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
            want = ol.linattn_forward(*make_inputs(wl, seed=seed), eps=wl.eps, rope=spec)
            got64 = got.float().cpu().double().numpy()
            assert float(np.max(np.abs(got64 - want)) / np.max(np.abs(want))) <= TOL


def test_noalloc_refuses_shapes_beyond_its_scratch(cuda_device):
    sla = _sla()
    lib = sla.raw_lib()
    wl = Workload("na_big", B=1, H=400, grid=(1, 1, 8))      # 400 heads: more than fits
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=15))
    out = torch.full_like(q, 7.0)
    stream = torch.cuda.current_stream(cuda_device)
    with torch.cuda.device(cuda_device):
        rc = lib.sla_linattn_forward_noalloc(*_args(q, k, v, g, out, None), None,
                                             stream.cuda_stream)
    torch.cuda.synchronize(cuda_device)
    assert rc == sla.UNSUPPORTED
    assert torch.all(out == 7.0)          # nothing ran
