"""Failure detection without a GPU fault: a bounded wait that runs out.

Every wait in the library's kernels gives up after a time limit, sets the device status
word and lets the kernel return.  ``sla_selftest_wait_timeout`` runs that path on purpose:
one thread waits on an mbarrier nobody arrives at, with the kernels' own wait and a limit
of about a millisecond.  The status must read SLA_ERR_DEVICE_TIMEOUT once, then SLA_OK
(the read clears it), and the device must stay usable: a forward right after it still
matches the oracle.
"""
import time

import numpy as np
import pytest

import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_wait_gives_up_and_reports_a_timeout(limit_us, cuda_device):
    sla = _sla()
    assert sla.last_device_status(device=cuda_device) == sla.OK
    t0 = time.perf_counter()
    sla.selftest_wait_timeout(limit_us, device=cuda_device)
    assert sla.last_device_status(device=cuda_device) == sla.DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed >= limit_us * 1e-6            # the wait lasted at least its limit
    assert sla.last_device_status(device=cuda_device) == sla.OK      # the read cleared it


def test_device_is_usable_after_a_timeout(cuda_device):
    sla = _sla()
    sla.selftest_wait_timeout(1000, device=cuda_device)
    assert sla.last_device_status(device=cuda_device) == sla.DEVICE_TIMEOUT
    wl = Workload("after_timeout", B=1, H=3, grid=(3, 9, 14), rope=True)
    host = make_inputs(wl, seed=41)
    q, k, v, g = (t.to(cuda_device) for t in host)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    for path in ("fused", "split"):
        with sla.forward_kernel(path):
            out = sla.linattn_forward(q, k, v, g, rope=rope, eps=wl.eps)
        assert sla.last_device_status(device=cuda_device) == sla.OK
        ref = ol.linattn_forward(*host, eps=wl.eps,
                                 rope=ol.RopeSpec(*wl.grid, *wl.split, base=wl.base))
        got = out.float().cpu().double().numpy()
        assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= wl.tol
