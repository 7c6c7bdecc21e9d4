"""Training without recomputing the state, through the C ABI:
sla_linattn_forward_keep_state (the forward that also writes each head's state)
and sla_linattn_backward_from_state (the backward that takes that state as its
S, z instead of summing them over k and v again).

- The output of the keeping forward is the plain forward's, bit for bit, under
  both launch plans.
- Its state: under the two-launch plan the very bytes sla_linattn_state writes;
  under the fused plan (the cluster's partials summed in rank order) S^T and z
  decoded from the documented layout match the oracle's S and z.
- The backward from sla_linattn_state's state equals the recomputing backward
  bit for bit; from the fused plan's state, it matches the backward oracle at
  the bf16 bound (max|err| / max|ref| <= 1e-2 per gradient).
"""
import numpy as np
import pytest
import torch

import oracle.backward as ob
import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

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


def _decode(state, B, H):
    """(S^T [B][H][128][128], z [B][H][128]) from the state layout: per head,
    S^T as bf16 in two 64-column halves of 128-byte rows whose 16-byte chunks
    are placed at chunk ^ (row % 8), then z as 128 fp32."""
    per = 32768 + 512
    st = np.empty((B, H, 128, 128))
    z = np.empty((B, H, 128))
    raw_all = state.cpu()
    for b in range(B):
        for h in range(H):
            base = (b * H + h) * per
            raw = raw_all[base:base + 32768].view(torch.bfloat16).float().numpy()
            raw = raw.reshape(2, 128, 8, 8)
            for half in range(2):
                for cpos in range(8):
                    rows = np.arange(128)
                    chunk = half * 8 + (cpos ^ (rows % 8))
                    for n in range(128):
                        st[b, h, n, chunk[n] * 8:(chunk[n] + 1) * 8] = raw[half, n, cpos]
            z[b, h] = raw_all[base + 32768:base + per].view(torch.float32).numpy()
    return st, z


CASES = [
    (1, 2, (1, 8, 16), True),
    (2, 3, (1, 1, 1000), False),
    (2, 4, (2, 9, 17), True),
    (1, 1, (4, 32, 32), True),       # 4096 tokens: the fused plan's widest clusters
    (1, 1, (1, 1, 1), True),         # one token
    (4, 50, (1, 4, 16), False),      # 200 heads, more than the SMs: the two launches
]


@pytest.mark.parametrize("plan", ["split", "fused"])
@pytest.mark.parametrize("B,H,grid,rope", CASES,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-{'rope' if r else 'norope'}"
                              for b, h, g, r in CASES])
def test_keep_state_and_backward_from_it(B, H, grid, rope, plan, cuda_device):
    sla = _sla()
    wl = Workload("keep", B=B, H=H, grid=grid, dtype=torch.bfloat16, rope=rope)
    tensors = _inputs(wl, seed=77)
    q, k, v, g, dout = (t.to(cuda_device) for t in tensors)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device) if rope else None
    with sla.forward_kernel(plan):
        want = sla.linattn_forward(q, k, v, g, rope=table, eps=wl.eps)
        out, state = sla.linattn_forward_keep_state(q, k, v, g, rope=table, eps=wl.eps)
        # the plan the calls took (the fused one does not apply to every shape)
        split = sla.forward_cluster(B, H, wl.N, rope, device=cuda_device) == 0
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, want)
    assert state.numel() == sla.state_bytes(B, H)

    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if rope else None
    if split:
        assert torch.equal(state, sla.linattn_state(k, v, rope=table))
    else:
        st, z = _decode(state, B, H)
        angles = ol.rope3d_angles(spec) if rope else None
        for b in range(B):
            for h in range(H):
                S_ref, z_ref = ol.linattn_state(_np64(tensors[1][b, h]), _np64(tensors[2][b, h]),
                                                angles)
                assert _rel(st[b, h], S_ref.T) <= 1e-2
                assert np.max(np.abs(z[b, h] - z_ref)) <= 1e-5 * np.max(np.abs(z_ref))

    got = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps, state=state)
    assert sla.last_device_status(device=cuda_device) == 0
    if split:
        ref = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps)
        for name, a, b in zip(NAMES, got, ref):
            assert torch.equal(a, b), name
    if wl.N == 1:
        # one token: dq = phi(k) (v . a) eps / den exactly, a difference of two terms of
        # size one that cancel to about eps, so the bf16 bound relative to max|ref| does
        # not apply; the bit-for-bit match with the recomputing backward above stands
        return
    ref = ob.linattn_backward(*tensors, eps=wl.eps, rope=spec)
    for name, a, b in zip(NAMES, got, ref):
        assert _rel(_np64(a), b) <= 1e-2, name


@pytest.mark.parametrize("name", ["5b_720p", "5b_480p"])
def test_training_step_full_size(name, cuda_device):
    """The forward keeping its state, then the backward from it, at full size:
    the output equals the plain forward's, and the gradients match the
    recomputing backward (bit for bit under the two-launch plan of 720p) and
    the oracle on sampled rows of two heads."""
    sla = _sla()
    wl = WORKLOADS[name]
    tensors = _inputs(wl, seed=0)
    q, k, v, g, dout = (t.to(cuda_device) for t in tensors)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device) if wl.rope else None
    want = sla.linattn_forward(q, k, v, g, rope=table, eps=wl.eps)
    out, state = sla.linattn_forward_keep_state(q, k, v, g, rope=table, eps=wl.eps)
    got = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps, state=state)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, want)
    del want, out
    if sla.forward_cluster(wl.B, wl.H, wl.N, wl.rope, device=cuda_device) == 0:
        ref = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps)
        for gname, a, b in zip(NAMES, got, ref):
            assert torch.equal(a, b), gname
        del ref
    rows = sample_rows(wl.N, 24)
    heads = [(0, 0), (1, wl.H - 1)]
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
    ref = ob.linattn_backward_rows(*tensors, rows, wl.eps, spec, heads)
    for i, gname in enumerate(NAMES):
        g_gpu = np.stack([_np64(got[i][b, h][rows]) for b, h in heads])
        g_ref = np.stack([ref[bh][i] for bh in heads])
        assert _rel(g_gpu, g_ref) <= wl.tol, gname


def test_keep_state_rejects_bad_buffers(cuda_device):
    """A state that overlaps an input or the output, or is misaligned, is refused
    before anything runs; so is a backward whose gradient overlaps the state."""
    sla = _sla()
    lib = sla.raw_lib()
    wl = Workload("bad", B=1, H=2, grid=(1, 1, 300), dtype=torch.bfloat16, rope=False)
    q, k, v, g, dout = (t.to(cuda_device) for t in _inputs(wl, seed=5))
    out = torch.empty_like(q)
    state = torch.empty(sla.state_bytes(1, 2) + 16, dtype=torch.uint8, device=cuda_device)
    B, H, N, d = q.shape
    stream = torch.cuda.current_stream(cuda_device).cuda_stream
    args = lambda st: (q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), out.data_ptr(),
                       B, H, N, d, None, 1e-6, st, stream)
    assert lib.sla_linattn_forward_keep_state(*args(None)) == sla.INVALID_ARG
    assert lib.sla_linattn_forward_keep_state(*args(k.data_ptr())) == sla.INVALID_ARG
    assert lib.sla_linattn_forward_keep_state(*args(out.data_ptr() + 64)) == sla.INVALID_ARG
    assert lib.sla_linattn_forward_keep_state(*args(state.data_ptr() + 8)) == sla.ALIGNMENT
    assert lib.sla_linattn_forward_keep_state(*args(state.data_ptr())) == sla.OK
    dq, dk, dv, dg = (torch.empty_like(q) for _ in range(4))
    bargs = lambda st, first: (q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                               dout.data_ptr(), st, first, dk.data_ptr(), dv.data_ptr(),
                               dg.data_ptr(), B, H, N, d, None, 1e-6, stream)
    assert lib.sla_linattn_backward_from_state(*bargs(None, dq.data_ptr())) == sla.INVALID_ARG
    assert lib.sla_linattn_backward_from_state(
        *bargs(state.data_ptr(), state.data_ptr())) == sla.INVALID_ARG
    assert lib.sla_linattn_backward_from_state(*bargs(state.data_ptr(), dq.data_ptr())) == sla.OK
    assert sla.last_device_status(device=cuda_device) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_autograd_function(dtype, cuda_device):
    """sla.linattn under torch autograd: its output is the forward's and its
    gradients the backward's (bit for bit; the two-launch plan for bf16, whose
    kept state is the recomputed one), and both meet the oracle."""
    sla = _sla()
    wl = Workload("autograd", B=2, H=3, grid=(2, 9, 17), dtype=dtype, rope=True)
    tensors = _inputs(wl, seed=91)
    q, k, v, g, dout = (t.to(cuda_device) for t in tensors)
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    leaves = [t.clone().requires_grad_() for t in (q, k, v, g)]
    with sla.forward_kernel("split"):
        out = sla.linattn(*leaves, rope=table, eps=wl.eps)
        want = sla.linattn_forward(q, k, v, g, rope=table, eps=wl.eps)
    out.backward(dout)
    ref = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out.detach(), want)
    for name, leaf, r in zip(NAMES, leaves, ref):
        assert torch.equal(leaf.grad, r), name
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base)
    tol = 1e-5 if dtype == torch.float32 else 1e-2
    for name, leaf, r in zip(NAMES, leaves, ob.linattn_backward(*tensors, eps=wl.eps, rope=spec)):
        assert _rel(_np64(leaf.grad), r) <= tol, name


def test_entries_from_a_thread_without_a_current_context(cuda_device):
    """Calls from a thread that has never made a CUDA context current (as a
    framework's backward worker may be; torch skips cudaSetDevice when the device
    number already matches), with the library's workspace already grown so that
    the call makes no allocation: the library binds the context itself, and the
    results equal the same calls made from this thread."""
    import threading
    sla = _sla()
    wl = Workload("thread", B=2, H=3, grid=(2, 9, 17), dtype=torch.bfloat16, rope=True)
    q, k, v, g, dout = (t.to(cuda_device) for t in _inputs(wl, seed=93))
    table = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    with sla.forward_kernel("split"):
        out, state = sla.linattn_forward_keep_state(q, k, v, g, rope=table, eps=wl.eps)
    want = sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps, state=state)
    fwd = sla.linattn_forward(q, k, v, g, rope=table, eps=wl.eps)
    torch.cuda.synchronize(cuda_device)
    got = [torch.empty_like(q) for _ in range(4)]
    got_fwd = torch.empty_like(q)
    errors = []

    def worker():
        try:
            sla.linattn_backward(q, k, v, g, dout, rope=table, eps=wl.eps, grads=got,
                                 state=state)
            sla.linattn_forward(q, k, v, g, out=got_fwd, rope=table, eps=wl.eps)
        except Exception as e:          # reported on the main thread
            errors.append(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert not errors, errors
    torch.cuda.synchronize(cuda_device)
    assert sla.last_device_status(device=cuda_device) == 0
    for name, a, b in zip(NAMES, got, want):
        assert torch.equal(a, b), name
    assert torch.equal(got_fwd, fwd)
