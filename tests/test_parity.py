"""CUDA path vs the fp64 oracle, through the C ABI.

Small shapes are compared element by element; they span several 128-token
tiles and a ragged tail.  The full-size workloads are compared on sampled
token rows: each head's state is formed by the oracle over all N tokens, the
outputs at the sampled rows are checked.  The bound is max|err| / max|ref|:
1e-5 for fp32 inputs, 1e-2 for bf16 inputs with fp32 accumulation.
"""
import numpy as np
import pytest
import torch

import oracle.linattn as ol
from gated_linear_attention_attn_b300.workloads import WORKLOADS, Workload, make_inputs, sample_rows

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2}


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


def _np64(t):
    return t.detach().float().cpu().double().numpy()


def _rel(out, ref):
    return float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))


def _spec(wl: Workload):
    return ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None


def _rope_table(wl: Workload, device):
    return _sla().RopeTable(wl.grid, wl.split, wl.base, device=device) if wl.rope else None


def _run(wl, tensors, device, path="auto"):
    q, k, v, g = (t.to(device) for t in tensors)
    with _sla().forward_kernel(path):
        out = _sla().linattn_forward(q, k, v, g, rope=_rope_table(wl, device), eps=wl.eps)
    assert _sla().last_device_status(device=device) == 0
    return out


SMALL = [
    # (B, H, grid, dtype, rope)
    (1, 1, (1, 1, 1), torch.bfloat16, False),
    (1, 2, (1, 1, 7), torch.bfloat16, True),
    (2, 3, (1, 1, 127), torch.bfloat16, False),
    (1, 2, (1, 8, 16), torch.bfloat16, True),
    (1, 2, (1, 1, 129), torch.bfloat16, False),
    (1, 3, (3, 10, 10), torch.bfloat16, True),
    (2, 2, (10, 10, 10), torch.bfloat16, True),
    (1, 2, (11, 15, 26), torch.bfloat16, False),
    (4, 16, (1, 1, 3), torch.bfloat16, True),
    (8, 32, (1, 1, 40), torch.bfloat16, False),     # 256 heads: more heads than SMs
    (2, 3, (1, 1, 1), torch.bfloat16, True),         # one token per head
    (1, 1, (2, 33, 31), torch.bfloat16, True),       # one head, 16 tiles and a ragged tail
    (1, 1, (5, 7, 9), torch.float32, True),
    (2, 3, (1, 1, 129), torch.float32, False),
    (1, 2, (4, 8, 8), torch.float32, True),
]


@pytest.mark.parametrize("path", ["fused", "split"])
@pytest.mark.parametrize("B,H,grid,dtype,rope", SMALL,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-{str(dt)[6:]}-{'rope' if r else 'norope'}"
                              for b, h, g, dt, r in SMALL])
def test_small_shapes_elementwise(B, H, grid, dtype, rope, path, cuda_device):
    """Both launch plans of the bf16 forward ("fused" falls back to the two
    launches where one head has a single 128-token tile)."""
    wl = Workload("small", B=B, H=H, grid=grid, dtype=dtype, rope=rope)
    tensors = make_inputs(wl, seed=7)
    out = _run(wl, tensors, cuda_device, path)
    ref = ol.linattn_forward(*tensors, eps=wl.eps, rope=_spec(wl))
    assert _rel(_np64(out), ref) <= TOL[dtype]


# Shapes whose fused plan takes each cluster size C = min(8, SMs // heads,
# 128-token tiles), lowered by the device where that many clusters do not fit
# at once; ragged tails in both tile sizes.
FUSED = [
    # (B, H, grid, rope, C expected on a 148-SM device)
    (2, 1, (1, 22, 50), True, 8),
    (1, 2, (1, 1, 891), False, 7),
    (1, 3, (7, 10, 10), True, 6),
    (1, 1, (1, 20, 30), False, 5),
    (2, 1, (5, 10, 10), True, 4),
    (3, 1, (1, 1, 300), False, 3),
    (1, 5, (2, 10, 10), True, 2),
    (1, 60, (1, 3, 100), True, 2),
]


@pytest.mark.parametrize("B,H,grid,rope,C", FUSED,
                         ids=[f"B{b}H{h}N{g[0]*g[1]*g[2]}-C{c}-{'rope' if r else 'norope'}"
                              for b, h, g, r, c in FUSED])
def test_fused_cluster_sizes_elementwise(B, H, grid, rope, C, cuda_device):
    sla = _sla()
    wl = Workload("fused", B=B, H=H, grid=grid, rope=rope)
    with sla.forward_kernel("fused"):
        got_c = sla.forward_cluster(B, H, wl.N, rope, device=cuda_device)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    assert 2 <= got_c <= min(8, sms // (B * H), (wl.N + 127) // 128)
    if sms == 148:
        assert got_c <= C
    tensors = make_inputs(wl, seed=17)
    out = _run(wl, tensors, cuda_device, "fused")
    ref = ol.linattn_forward(*tensors, eps=wl.eps, rope=_spec(wl))
    assert _rel(_np64(out), ref) <= TOL[torch.bfloat16]
    split = _run(wl, tensors, cuda_device, "split")
    assert _rel(_np64(out), _np64(split)) <= TOL[torch.bfloat16]


def test_plan_choice_follows_the_override(cuda_device):
    sla = _sla()
    with sla.forward_kernel("split"):
        assert sla.forward_cluster(2, 20, 4290, False, device=cuda_device) == 0
    with sla.forward_kernel("fused"):
        assert sla.forward_cluster(1, 1, 128, False, device=cuda_device) == 0   # one tile
        assert sla.forward_cluster(1, 200, 4096, False, device=cuda_device) == 0  # too many heads
        assert sla.forward_cluster(2, 20, 4290, False, device=cuda_device) >= 2


def test_tiny_fp32_workload_elementwise(cuda_device):
    wl = WORKLOADS["tiny_fp32"]
    tensors = make_inputs(wl, seed=0)
    out = _run(wl, tensors, cuda_device)
    ref = ol.linattn_forward(*tensors, eps=wl.eps, rope=_spec(wl))
    assert _rel(_np64(out), ref) <= 1e-5


_FULL_CACHE = {}


def _full_size_case(name):
    """Inputs, sampled rows, heads and the oracle's rows for a workload (kept
    for the other launch plan)."""
    if name not in _FULL_CACHE:
        wl = WORKLOADS[name]
        tensors = make_inputs(wl, seed=0)
        rows = sample_rows(wl.N, 48)
        heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
        if wl.N > 50000:          # the longest clip: first, last and two more heads
            heads = [heads[0], heads[7], heads[13], heads[-1]]
        q, k, v, g = tensors
        ref = ol.linattn_forward_rows(q, k, v, g, rows, eps=wl.eps, rope=_spec(wl), heads=heads)
        _FULL_CACHE.clear()
        _FULL_CACHE[name] = (tensors, rows, heads, np.stack([ref[bh] for bh in heads]))
    return _FULL_CACHE[name]


@pytest.mark.parametrize("path", ["auto", "split"])
@pytest.mark.parametrize("name", ["5b_480p", "5b_720p", "14b_480p", "5b_720p_60s",
                                  "5b_720p_736"])
def test_full_size_sampled_rows(name, path, cuda_device):
    """"auto" is the plan the benchmark times."""
    wl = WORKLOADS[name]
    tensors, rows, heads, want = _full_size_case(name)
    out = _run(wl, tensors, cuda_device, path)
    got = np.stack([_np64(out[b, h][rows]) for b, h in heads])
    assert _rel(got, want) <= wl.tol
    assert np.all(np.isfinite(_np64(out[0, 0])))


def test_shapes_and_plans_alternate_on_one_stream(cuda_device):
    """One stream's workspace serves calls of every shape and plan: each call's per-head
    counters must start at zero although a call of another shape may have left partial
    states where they lie.  Each (shape, plan) must give its first result bit for bit
    every time, and match the oracle."""
    sla = _sla()
    shapes = [Workload("alt_a", B=2, H=50, grid=(1, 10, 60), rope=True),     # 100 heads
              Workload("alt_b", B=1, H=64, grid=(1, 4, 100), rope=False),    # 64 heads
              Workload("alt_c", B=1, H=3, grid=(3, 10, 20), rope=True)]
    first = {}
    order = [(0, "split"), (1, "split"), (2, "fused"), (0, "split"), (2, "split"),
             (1, "fused"), (0, "split"), (1, "split"), (2, "split"), (0, "fused")]
    inputs = {i: make_inputs(wl, seed=50 + i) for i, wl in enumerate(shapes)}
    for i, path in order:
        wl = shapes[i]
        out = _run(wl, inputs[i], cuda_device, path)
        key = (i, path)
        if key not in first:
            first[key] = out
            ref = ol.linattn_forward(*inputs[i], eps=wl.eps, rope=_spec(wl))
            assert _rel(_np64(out), ref) <= TOL[torch.bfloat16], key
        else:
            assert torch.equal(out, first[key]), key


def test_dead_query_rows_are_zero(cuda_device):
    wl = Workload("dead", B=1, H=2, grid=(3, 10, 10), rope=True)
    q, k, v, g = make_inputs(wl, seed=3)
    q[:, :, 5] = -q[:, :, 5].abs() - 0.1         # phi(q) = 0: num = 0, den = eps
    q[:, :, 299] = -1.0
    out = _run(wl, (q, k, v, g), cuda_device)
    assert torch.all(out[:, :, 5] == 0) and torch.all(out[:, :, 299] == 0)


def test_constant_values_pass_through(cuda_device):
    wl = Workload("const", B=1, H=2, grid=(2, 20, 20), rope=False)
    q, k, _, _ = make_inputs(wl, seed=4)
    c = torch.linspace(-2, 2, 128).to(torch.bfloat16)
    v = c.expand(1, 2, wl.N, 128).contiguous()
    g = torch.full_like(q, 40.0)
    out = _run(wl, (q, k, v, g), cuda_device)
    err = (out.float().cpu() - c.float()).abs().max().item()
    assert err <= 1e-2 * c.float().abs().max().item()


def test_large_eps_and_saturated_gate(cuda_device):
    wl = Workload("eps", B=1, H=2, grid=(1, 9, 30), rope=True, eps=5.0)
    q, k, v, _ = make_inputs(wl, seed=5)
    g = torch.full_like(q, 40.0)
    out = _run(wl, (q, k, v, g), cuda_device)
    ref = ol.linattn_forward(q, k, v, g, eps=5.0, rope=_spec(wl))
    assert _rel(_np64(out), ref) <= 1e-2


def test_repeatable_and_stream_independent(cuda_device):
    wl = Workload("rep", B=2, H=3, grid=(4, 11, 13), rope=True)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=6))
    rope = _rope_table(wl, cuda_device)
    sla = _sla()
    a = sla.linattn_forward(q, k, v, g, rope=rope)
    b = sla.linattn_forward(q, k, v, g, rope=rope)
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(s):
        c = sla.linattn_forward(q, k, v, g, rope=rope)
    s.synchronize()
    torch.cuda.synchronize(cuda_device)
    assert torch.equal(a, b) and torch.equal(a, c)


def test_phases_equal_forward(cuda_device):
    """sla_linattn_state + sla_linattn_apply give the two-launch forward's
    output bit for bit."""
    sla = _sla()
    for rope_on in (False, True):
        wl = Workload("phases", B=2, H=3, grid=(3, 7, 11), rope=rope_on)
        q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=8))
        rope = _rope_table(wl, cuda_device)
        with sla.forward_kernel("split"):
            fwd = sla.linattn_forward(q, k, v, g, rope=rope)
        state = sla.linattn_state(k, v, rope=rope)
        out = sla.linattn_apply(q, g, state, rope=rope)
        assert sla.last_device_status(device=cuda_device) == 0
        assert torch.equal(fwd, out)
        assert state.numel() == sla.state_bytes(2, 3) == 6 * 33280


def test_apply_with_other_queries(cuda_device):
    """A state of one token set applied to queries of another (own grids, own RoPE)."""
    sla = _sla()
    wk = Workload("keys", B=1, H=2, grid=(4, 6, 10), rope=True)
    wq = Workload("queries", B=1, H=2, grid=(2, 5, 13), rope=True)
    _, k, v, _ = make_inputs(wk, seed=9)
    q, _, _, g = make_inputs(wq, seed=10)
    rk, rq = _rope_table(wk, cuda_device), _rope_table(wq, cuda_device)
    state = sla.linattn_state(k.to(cuda_device), v.to(cuda_device), rope=rk)
    out = sla.linattn_apply(q.to(cuda_device), g.to(cuda_device), state, rope=rq)
    assert sla.last_device_status(device=cuda_device) == 0
    ak, aq = ol.rope3d_angles(_spec(wk)), ol.rope3d_angles(_spec(wq))
    ref = np.empty((1, 2, wq.N, 128))
    for h in range(2):
        S, z = ol.linattn_state(_np64(k[0, h]), _np64(v[0, h]), ak)
        ref[0, h] = ol.linattn_apply(_np64(q[0, h]), _np64(g[0, h]), S, z, 1e-6, aq)
    assert _rel(_np64(out), ref) <= 1e-2


def test_state_layout_holds_s_and_z(cuda_device):
    """The documented state layout: S^T in bf16 (swizzled chunks), then z in fp32."""
    sla = _sla()
    wl = Workload("layout", B=1, H=1, grid=(1, 3, 100), rope=False)
    _, k, v, _ = make_inputs(wl, seed=12)
    state = sla.linattn_state(k.to(cuda_device), v.to(cuda_device)).cpu()
    S, z = ol.linattn_state(_np64(k[0, 0]), _np64(v[0, 0]))
    raw = state[:32768].view(torch.bfloat16).float().numpy().reshape(2, 128, 8, 8)
    st = np.empty((128, 128))                      # S^T[n][m]
    for n in range(128):
        for cpos in range(8):
            for half in range(2):
                chunk = half * 8 + (cpos ^ (n % 8))
                st[n, chunk * 8:(chunk + 1) * 8] = raw[half, n, cpos]
    assert _rel(st, S.T) <= 1e-2
    zz = state[32768:33280].view(torch.float32).numpy()
    assert np.max(np.abs(zz - z)) <= 1e-5 * np.max(np.abs(z))
