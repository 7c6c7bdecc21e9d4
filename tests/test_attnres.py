"""AttnRes aggregation, CUDA path vs the fp64 oracle (oracle/attnres.py),
through the C ABI (sla_attnres_aggregate).

Small shapes are compared element by element (one to eight sources, hidden
sizes 256 to 4096, token counts that do not fill the last block of warps);
the full-size workloads on sampled tokens.  The bound is
max|err| / max|ref| <= 1e-2 (bf16 in and out, fp32 arithmetic).
"""
import numpy as np
import pytest
import torch

import oracle.attnres as oa
from gated_linear_attention_attn_b300.workloads import (WORKLOADS, Workload, make_attnres_inputs,
                                                        sample_rows)

pytestmark = pytest.mark.gpu

TOL = 1e-2
EPS = 1e-6


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _rel(out, ref):
    return float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))


def _wl(M, T, C):
    return Workload("attnres", B=1, H=M, grid=(1, 1, T), d=C, layer="attnres")


CASES = [(1, 1, 256), (2, 7, 256), (4, 13, 2560), (5, 9, 4096), (8, 17, 512), (3, 100, 768),
         # more than 384 threads a CTA: rows held in bf16 (M <= 5) or read again (M > 5),
         # and more tokens than resident CTAs, so that every slot is refilled
         (1, 5, 4096), (2, 50, 3328), (5, 1500, 4096), (6, 9, 3584), (8, 700, 4096)]


@pytest.mark.parametrize("M,T,C", CASES, ids=[f"M{m}T{t}C{c}" for m, t, c in CASES])
def test_attnres_elementwise(M, T, C, cuda_device):
    s, w = make_attnres_inputs(_wl(M, T, C), seed=11)
    got = _sla().attnres_aggregate(s.to(cuda_device), w.to(cuda_device), eps=EPS)
    want = oa.attnres_aggregate(s.double().numpy(), w.double().numpy(), EPS)
    assert _rel(got.double().cpu().numpy(), want) <= TOL


def test_attnres_list_of_sources_and_zero_query(cuda_device):
    s, w = make_attnres_inputs(_wl(3, 40, 512), seed=12)
    parts = [x.to(cuda_device).contiguous() for x in s.unbind(0)]
    got = _sla().attnres_aggregate(parts, torch.zeros_like(w).to(cuda_device), eps=EPS)
    want = s.double().mean(dim=0).numpy()
    assert _rel(got.double().cpu().numpy(), want) <= TOL


@pytest.mark.parametrize("name", ["attnres_5b_720p", "attnres_14b_480p"])
def test_attnres_full_size_sampled_tokens(name, cuda_device):
    wl = WORKLOADS[name]
    s, w = make_attnres_inputs(wl, seed=0)
    got = _sla().attnres_aggregate(s.to(cuda_device), w.to(cuda_device), eps=EPS)
    rows = sample_rows(wl.tokens, 64)
    want = oa.attnres_aggregate(s[:, rows].double().numpy(), w.double().numpy(), EPS)
    assert _rel(got[rows].double().cpu().numpy(), want) <= TOL
    assert torch.isfinite(got.float()).all()


def test_attnres_hidden_sizes_alternate(cuda_device):
    """One kernel (same source count, same rows-in-registers choice) launched with
    different shared-memory sizes in turn: a larger size after a smaller one must still
    launch (the kernel's shared-memory limit is not lowered by a smaller call)."""
    sla = _sla()
    for C in (2560, 512, 1024, 2560, 256, 2560):
        s, w = make_attnres_inputs(_wl(4, 33, C), seed=13)
        got = sla.attnres_aggregate(s.to(cuda_device), w.to(cuda_device), eps=EPS)
        assert sla.last_device_status(device=cuda_device) == sla.OK
        want = oa.attnres_aggregate(s.double().numpy(), w.double().numpy(), EPS)
        assert _rel(got.double().cpu().numpy(), want) <= TOL, C
