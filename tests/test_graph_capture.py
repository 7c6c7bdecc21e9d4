"""The bf16 entry points inside a captured CUDA graph.

A serving loop replays a captured graph instead of launching each call.  The
library's workspace is allocated on the first call of a shape, so one call
runs before capture; the captured replay must then give the call's result bit
for bit, for each launch plan and for the block-causal form.  The allocation-
free entry point only needs its first call on the device (which looks up its
scratch array) before capture.
"""
import ctypes

import pytest
import torch

from gated_linear_attention_attn_b300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _sla():
    from gated_linear_attention_attn_b300 import sla
    return sla


@pytest.mark.parametrize("path", ["fused", "split"])
def test_forward_replays_in_a_graph(path, cuda_device, monkeypatch):
    sla = _sla()
    monkeypatch.setenv("SLA_FORWARD_KERNEL", path)
    wl = Workload("graph", B=2, H=4, grid=(3, 10, 20), rope=True)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=31))
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    ref = sla.linattn_forward(q, k, v, g, rope=rope)        # allocates the workspace
    out = torch.full_like(q, float("nan"))
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        sla.linattn_forward(q, k, v, g, out=out, rope=rope, stream=stream)   # this stream's workspace
    stream.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.linattn_forward(q, k, v, g, out=out, rope=rope, stream=stream)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("path", ["split"])
def test_forward_replays_with_new_inputs(path, cuda_device, monkeypatch):
    """Every head spans many CTAs of the state kernel, whose shared merge counts the
    contributors in a per-head counter.  A replay reuses the captured launch's
    parameters, so the counters must be back at zero when a launch ends: with inputs
    changed between replays, each replay must give the eager call's result for its own
    inputs, bit for bit."""
    sla = _sla()
    monkeypatch.setenv("SLA_FORWARD_KERNEL", path)
    wl = Workload("graph_multi", B=2, H=4, grid=(4, 10, 110), rope=True)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=36))
    out = torch.empty_like(q)
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        sla.linattn_forward(q, k, v, g, out=out, rope=rope, stream=stream)  # workspace
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.linattn_forward(q, k, v, g, out=out, rope=rope, stream=stream)
    for seed in (37, 38, 39):
        fresh = [t.to(cuda_device) for t in make_inputs(wl, seed=seed)]
        with torch.cuda.stream(stream):
            for dst, src in zip((q, k, v, g), fresh):
                dst.copy_(src)
            graph.replay()
            ref = sla.linattn_forward(*fresh, rope=rope, stream=stream)
        stream.synchronize()
        assert sla.last_device_status(stream, device=cuda_device) == 0
        assert torch.equal(out, ref), seed


@pytest.mark.parametrize("path", ["split"])
def test_noalloc_replays_with_new_inputs(path, cuda_device, monkeypatch):
    """The same for the allocation-free entry point, whose counters live in its fixed
    array."""
    sla = _sla()
    lib = sla.raw_lib()
    monkeypatch.setenv("SLA_FORWARD_KERNEL", path)
    wl = Workload("graph_multi_na", B=2, H=4, grid=(4, 10, 110), rope=True)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=40))
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    B, H, N, d = q.shape
    stream = torch.cuda.Stream(cuda_device)

    def call():
        return lib.sla_linattn_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               g.data_ptr(), out.data_ptr(), B, H, N, d,
                                               rope.ptr, 1e-6, status.data_ptr(),
                                               stream.cuda_stream)

    with torch.cuda.device(cuda_device):
        assert call() == sla.OK               # looks up the array's address, outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        assert call() == sla.OK
    for seed in (41, 42, 43):
        fresh = [t.to(cuda_device) for t in make_inputs(wl, seed=seed)]
        with torch.cuda.stream(stream):
            for dst, src in zip((q, k, v, g), fresh):
                dst.copy_(src)
            graph.replay()
            ref = sla.linattn_forward(*fresh, rope=rope, stream=stream)
        stream.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref), seed


def test_block_causal_replays_in_a_graph(cuda_device):
    sla = _sla()
    wl = Workload("graphbc", B=1, H=3, grid=(4, 8, 10), rope=True, block_frames=2)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=32))
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        ref, st_ref = sla.linattn_forward_block_causal(q, k, v, g, wl.block_tokens, rope=rope,
                                                       stream=stream)
    stream.synchronize()
    out = torch.full_like(q, float("nan"))
    st = torch.full_like(st_ref, float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.linattn_forward_block_causal(q, k, v, g, wl.block_tokens, out=out, rope=rope,
                                         state_out=st, stream=stream)
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, ref) and torch.equal(st, st_ref)


def test_noalloc_replays_in_a_graph(cuda_device):
    sla = _sla()
    lib = sla.raw_lib()
    wl = Workload("graphna", B=1, H=2, grid=(2, 9, 11), rope=False)
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=33))
    ref = sla.linattn_forward(q, k, v, g)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    B, H, N, d = q.shape
    stream = torch.cuda.Stream(cuda_device)
    # the device address of the scratch array is looked up once per device, outside capture
    with torch.cuda.device(cuda_device):
        rc = lib.sla_linattn_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             g.data_ptr(), out.data_ptr(), B, H, N, d, None,
                                             1e-6, status.data_ptr(), stream.cuda_stream)
    assert rc == sla.OK
    stream.synchronize()
    out.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        rc = lib.sla_linattn_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             g.data_ptr(), out.data_ptr(), B, H, N, d, None,
                                             1e-6, status.data_ptr(), stream.cuda_stream)
    assert rc == sla.OK
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert int(status.item()) == 0
    assert torch.equal(out, ref)


def test_anchor_replays_in_a_graph(cuda_device):
    """The anchor forward (RoPE pre-pass into the stream's workspace, then the
    attention kernel) replays bit for bit."""
    sla = _sla()
    wl = Workload("graphan", B=1, H=2, grid=(2, 8, 20), d=256, rope=True, split=(88, 84, 84),
                  layer="anchor")
    q, k, v, g = (t.to(cuda_device) for t in make_inputs(wl, seed=34))
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        ref = sla.anchor_forward(q, k, v, g, rope=rope, stream=stream)   # this stream's workspace
    stream.synchronize()
    out = torch.full_like(q, float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.anchor_forward(q, k, v, g, out=out, rope=rope, stream=stream)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, ref)


def test_attnres_replays_in_a_graph(cuda_device):
    from gated_linear_attention_attn_b300.workloads import make_attnres_inputs
    sla = _sla()
    wl = Workload("graphar", B=1, H=4, grid=(1, 1, 300), d=2560, layer="attnres")
    s, w = (t.to(cuda_device) for t in make_attnres_inputs(wl, seed=35))
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        ref = sla.attnres_aggregate(s, w, stream=stream)
    stream.synchronize()
    out = torch.full_like(ref, float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.attnres_aggregate(s, w, out=out, stream=stream)
    graph.replay()
    torch.cuda.synchronize(cuda_device)
    assert sla.last_device_status(device=cuda_device) == 0
    assert torch.equal(out, ref)


def test_backward_replays_with_new_inputs(cuda_device):
    """The bf16 backward's six launches, each after the first a programmatic dependent of
    the one before, captured into one graph: with new inputs copied into the captured
    buffers before each replay, every replay gives the eager call's gradients for those
    inputs, bit for bit (heads span several CTAs, so the state kernel's counters and the
    dS and dz partial slots are all used)."""
    sla = _sla()
    wl = Workload("graph_bwd", B=2, H=4, grid=(4, 10, 110), rope=True)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)

    def inputs(seed):
        q, k, v, g = make_inputs(wl, seed=seed)
        gen = torch.Generator().manual_seed(seed + 1000)
        dout = torch.randn(q.shape, generator=gen).to(wl.dtype)
        return [t.to(cuda_device) for t in (q, k, v, g, dout)]

    bufs = inputs(36)
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(stream):
        sla.linattn_backward(*bufs, rope=rope, stream=stream)      # this stream's workspace
    stream.synchronize()
    grads = [torch.full_like(bufs[0], float("nan")) for _ in range(4)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        sla.linattn_backward(*bufs, rope=rope, grads=grads, stream=stream)
    for seed in (37, 38):
        new = inputs(seed)
        with torch.cuda.stream(stream):
            for dst, src in zip(bufs, new):
                dst.copy_(src)
            graph.replay()
            want = sla.linattn_backward(*new, rope=rope, stream=stream)
        stream.synchronize()
        assert sla.last_device_status(device=cuda_device) == 0
        for name, a, b in zip(("dq", "dk", "dv", "dg"), grads, want):
            assert torch.equal(a, b), (seed, name)


@pytest.mark.parametrize("path", ["split", "fused"])
def test_training_step_replays_with_new_inputs(path, cuda_device):
    """One training step (the forward keeping its state, then the backward from it:
    seven or six launches) captured into one graph: with new inputs and upstream
    gradient copied in before each replay, every replay gives the eager step's output
    and gradients for those inputs, bit for bit, under both forward plans."""
    sla = _sla()
    wl = Workload("graph_train", B=2, H=4, grid=(4, 10, 110), rope=True)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=cuda_device)

    def inputs(seed):
        q, k, v, g = make_inputs(wl, seed=seed)
        gen = torch.Generator().manual_seed(seed + 1000)
        dout = torch.randn(q.shape, generator=gen).to(wl.dtype)
        return [t.to(cuda_device) for t in (q, k, v, g, dout)]

    def step(bufs, out, state, grads, stream):
        q, k, v, g, dout = bufs
        sla.linattn_forward_keep_state(q, k, v, g, out=out, rope=rope, state=state,
                                       stream=stream)
        sla.linattn_backward(q, k, v, g, dout, rope=rope, grads=grads, stream=stream,
                             state=state)

    bufs = inputs(46)
    out = torch.full_like(bufs[0], float("nan"))
    state = torch.zeros(sla.state_bytes(wl.B, wl.H), dtype=torch.uint8, device=cuda_device)
    grads = [torch.full_like(bufs[0], float("nan")) for _ in range(4)]
    stream = torch.cuda.Stream(cuda_device)
    stream.wait_stream(torch.cuda.current_stream(cuda_device))
    with sla.forward_kernel(path):
        with torch.cuda.stream(stream):
            step(bufs, out, state, grads, stream)                 # this stream's workspace
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step(bufs, out, state, grads, stream)
        for seed in (47, 48):
            new = inputs(seed)
            w_out = torch.empty_like(out)
            w_state = torch.empty_like(state)
            w_grads = [torch.empty_like(out) for _ in range(4)]
            with torch.cuda.stream(stream):
                for dst, src in zip(bufs, new):
                    dst.copy_(src)
                graph.replay()
                step(new, w_out, w_state, w_grads, stream)
            stream.synchronize()
            assert sla.last_device_status(device=cuda_device) == 0
            assert torch.equal(out, w_out), seed
            assert torch.equal(state, w_state), seed
            for name, a, b in zip(("dq", "dk", "dv", "dg"), grads, w_grads):
                assert torch.equal(a, b), (seed, name)
