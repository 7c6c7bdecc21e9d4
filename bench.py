"""Throughput of the gated linear-attention forward on synthetic latent-grid inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl sla|reference]

One step is one forward (state reduction + apply, every head) over the whole
workload, inputs already resident in HBM.  The metric is token-heads per
second (B*H*N / step time); the roofline object gives the achieved HBM
bandwidth of the dominant kernel against the measured peak.  Prints one JSON
line on rank 0.  Under torchrun each rank runs its own replica on its own GPU
(the heads are independent; nothing is exchanged), so `value` is the sum over
ranks of the work divided by the slowest rank's time.

`--impl reference` times the fp64 CPU oracle instead (one head of the
workload per step, on the host cores), for the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_linear_attention_attn_b300.workloads import HEADLINE, WORKLOADS, make_inputs  # noqa: E402

METRIC = "linear-attn fwd token-heads/s; HBM GB/s as % of B300 peak (5B 720p shape)"
UNIT = "token-heads/s"
FALLBACK_HBM_GBS = 6400.0
L2_BYTES = 126 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="sla", choices=["sla", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the oracle on the host")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-workloads", action="store_true",
                    help="on the headline workload, skip timing the other configurations")
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"],
                    help="time the layer's forward (the headline) or its backward")
    ap.add_argument("--forward-kernel", default="auto", choices=["auto", "fused", "split"],
                    help="launch plan of the bf16 forward (SLA_FORWARD_KERNEL)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            data = json.load(fh)
        return float(data["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while the GPU works.

    NVML is called through ctypes on the driver's libnvidia-ml.so.1; the GPU
    is matched to the CUDA device by PCI bus id.
    """

    REASONS = {0x2: "applications_clocks", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock"}
    NVML_CLOCK_SM = 1

    def __init__(self, device: torch.device, period_s: float = 0.002):
        import ctypes
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self.regions = 0
        self._stop = threading.Event()
        self._active = threading.Event()
        self._period = period_s
        self._thread = None
        self.error = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            bus = ctypes.create_string_buffer(64)
            cudart = ctypes.CDLL("libcudart.so.13")
            if cudart.cudaDeviceGetPCIBusId(bus, 64, int(device.index or 0)) != 0:
                raise RuntimeError("cudaDeviceGetPCIBusId failed")
            self._h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.value, ctypes.byref(self._h)) != 0:
                raise RuntimeError(f"no NVML handle for {bus.value!r}")
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(self._h, self.NVML_CLOCK_SM, ctypes.byref(mx))
            self.max_mhz = mx.value
            self._nv, self._ct = nv, ctypes
            self.sample()
        except Exception as exc:  # no NVML: report why instead of clocks
            self._nv = None
            self.error = repr(exc)

    def sample(self):
        ct, nv = self._ct, self._nv
        clk, bits = ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(self._h, self.NVML_CLOCK_SM, ct.byref(clk)) == 0:
            self.samples.append(clk.value)
        if nv.nvmlDeviceGetCurrentClocksEventReasons(self._h, ct.byref(bits)) == 0:
            for bit, name in self.REASONS.items():
                if bits.value & bit:
                    self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            if self._active.is_set():
                self.sample()
            time.sleep(self._period)

    def start(self):
        """Start the sampling thread; it samples only inside `timed()` regions."""
        if self._nv is not None:
            self.samples.clear()
            self.reasons.clear()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    class _Region:
        def __init__(self, owner):
            self.owner = owner

        def __enter__(self):
            if self.owner._nv is not None:
                self.owner.sample()
            self.owner._active.set()

        def __exit__(self, *exc):
            self.owner._active.clear()
            if self.owner._nv is not None:
                self.owner.sample()
            self.owner.regions += 1
            return False

    def timed(self):
        return ClockSampler._Region(self)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._nv is None:
            return {"error": self.error or "NVML unavailable"}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "timed_regions": self.regions, "reasons": sorted(self.reasons),
                "note": "sampled every %.0f ms inside every timed region of this run"
                        % (1e3 * self._period)}


# The sources each profiled kernel is built from.
_COMMON_SOURCES = ("tc_ptx.cuh", "common.cuh", "launch.h")
KERNEL_SOURCES = {
    "tc_state_kernel": ("tc_forward.cu", "tc_common.cuh") + _COMMON_SOURCES,
    "tc_apply_kernel": ("tc_forward.cu", "tc_common.cuh") + _COMMON_SOURCES,
    "tc_fused_kernel": ("tc_forward.cu", "tc_common.cuh") + _COMMON_SOURCES,
    "anchor_attn_kernel": ("anchor.cu",) + _COMMON_SOURCES,
    "attnres_kernel": ("attnres.cu",) + _COMMON_SOURCES,
}


def source_hash(kernel: str):
    """Hash of a kernel's sources, to tell whether a stored ncu traffic figure is current."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "gated_linear_attention_attn_b300", "csrc", name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/dram_traffic.txt, if taken on the current sources.

    Lines: `<kernel> <workload> <bytes_per_launch> <hash of the kernel's sources>`.
    """
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    current = source_hash(kernel)
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[3] == current:
                return float(parts[2])
    return None


# ------------------------------------------------------------ CPU oracle ----

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 0) for p in threadpool_info() if p.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_heads(wl, tensors, heads):
    """Run the fp64 oracle on the given (b, h) heads at full N; returns elapsed seconds."""
    import oracle.block_causal as bc   # the CPU baseline is the one place bench.py runs the oracle
    import oracle.linattn as ol
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
    q, k, v, g = tensors
    t0 = time.perf_counter()
    for b, h in heads:
        ang = ol.rope3d_angles(spec) if spec is not None else None
        args = (q[b, h].double().numpy(), k[b, h].double().numpy(), v[b, h].double().numpy(),
                g[b, h].double().numpy())
        if wl.block_frames:
            bc.linattn_block_causal_head(*args, wl.block_tokens, wl.eps, ang)
        else:
            ol.linattn_head(*args, wl.eps, ang)
    return time.perf_counter() - t0


def cpu_baseline(wl, tensors, budget_s=10.0):
    """The oracle as it stands on the host cores: heads of the workload, one after another,
    until about `budget_s` seconds have passed (at least one head)."""
    all_heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < 4 * len(all_heads):
        elapsed += oracle_heads(wl, tensors, [all_heads[done % len(all_heads)]])
        done += 1
    return {"value": done * wl.N / elapsed, "unit": UNIT, "cores": _blas_threads(),
            "kind": "oracle",
            "sample": f"{done} heads of {wl.name} at full N={wl.N} (fp64 numpy, "
                      f"{elapsed:.1f} s); token-heads = heads x N"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle on the host, one head of the workload per step."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    tensors = make_inputs(wl, seed=0)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    for i in range(args.warmup):
        oracle_heads(wl, tensors, [heads[i % len(heads)]])
    total = 0.0
    for i in range(args.steps):
        total += oracle_heads(wl, tensors, [heads[i % len(heads)]])
    value = args.steps * wl.N / total
    cores = _blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, world),
        "note": "one head (full N) per step on the host cores",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} heads of {wl.name}, one per step, full N"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def _config(wl, world):
    cfg = {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
           "grid": list(wl.grid), "rope": wl.rope,
           "rope_split": list(wl.split) if wl.rope else None, "eps": wl.eps,
           "k_scale": wl.k_scale, "input_dtype": str(wl.dtype).replace("torch.", ""),
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": ("inputs larger than L2 (%.0f MB vs 126 MB), steps back to back"
                  % (wl.algorithmic_bytes / 1e6) if wl.algorithmic_bytes >= 4 * L2_BYTES
                  else "L2 flushed between steps (a 252 MB buffer written, then "
                       "another read, outside the timed events)")}
    if wl.block_frames:
        cfg["block_frames"] = wl.block_frames
        cfg["block_tokens"] = wl.block_tokens
    if wl.layer == "anchor":              # softmax attention: no eps, keys unscaled
        cfg["layer"] = "gated-softmax anchor"
        del cfg["eps"], cfg["k_scale"]
    return cfg


# ------------------------------------------------------------------ GPU -----

def _max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


SAMPLER = None      # the run's ClockSampler; every timed region is sampled


def _start_sampler(dev):
    global SAMPLER
    SAMPLER = ClockSampler(dev)
    SAMPLER.start()


def _stop_sampler():
    """The clock record over every timed region so far (then sampling stops)."""
    global SAMPLER
    if SAMPLER is None:
        return {"error": "no timed region"}
    rec = SAMPLER.stop()
    SAMPLER = None
    return rec


def _time_steps(fn, steps, stream, flush=None):
    """Device seconds of `steps` calls of fn on `stream`: one event pair around
    all of them, or, with an L2 flush between steps, one pair per step with the
    flush outside the pairs."""
    if SAMPLER is not None:
        with SAMPLER.timed():
            return _time_steps_raw(fn, steps, stream, flush)
    return _time_steps_raw(fn, steps, stream, flush)


def _time_steps_raw(fn, steps, stream, flush=None):
    if flush is None:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            fn()
        t1.record(stream)
        t1.synchronize()
        return t0.elapsed_time(t1) / 1e3
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    evs[-1][1].synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3


class L2Scrub:
    """Evicts the previous step's data from L2 between timed steps, outside the events.

    A buffer of twice the L2 size is written, then a second one of that size is read: the
    L2 is left holding clean lines, so the write-back of the dirty ones (the previous
    step's outputs, the written buffer) happens here and not inside the next timed step.
    """

    def __init__(self, dev):
        self.written = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.read = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.written.fill_(1)
        torch.sum(self.read, dim=0, out=self.sink)


E2E_NOTE = ("pinned host buffers, two device buffer sets: every step uploads its inputs, runs the "
            "call and reads its outputs back; the upload of step i+1 overlaps the read-back of "
            "step i (the host link is full duplex)")


def pipelined_e2e(dev, stream, ke, dev_ins, host_ins, dev_outs, run):
    """Device seconds of ke end-to-end steps, their bytes in and out.

    Each step copies host_ins (pinned) to a set of device inputs on an upload stream, runs
    run(inputs, outputs) on `stream`, and copies the outputs back to pinned host buffers on a
    download stream. Two sets of device buffers alternate, so that one step's upload overlaps
    the previous step's read-back; every step still moves all of its own bytes.
    """
    ins = [list(dev_ins), [torch.empty_like(t) for t in dev_ins]]
    outs = [list(dev_outs), [torch.empty_like(t) for t in dev_outs]]
    houts = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_outs]
             for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded, computed, read = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def one(i):
        sl = i & 1
        if i >= 2:
            up.wait_event(computed[sl])          # step i - 2 has consumed these inputs
        with torch.cuda.stream(up):
            for d, h in zip(ins[sl], host_ins):
                d.copy_(h, non_blocking=True)
        uploaded[sl].record(up)
        stream.wait_event(uploaded[sl])
        if i >= 2:
            stream.wait_event(read[sl])          # and its outputs are read back
        run(ins[sl], outs[sl])
        computed[sl].record(stream)
        down.wait_event(computed[sl])
        with torch.cuda.stream(down):
            for h, d in zip(houts[sl], outs[sl]):
                h.copy_(d, non_blocking=True)
        read[sl].record(down)

    for i in range(2):
        one(i)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed():
        t0.record(up)
        for i in range(ke):
            one(i)
        t1.record(down)
        t1.synchronize()

    if SAMPLER is not None:
        with SAMPLER.timed():
            timed()
    else:
        timed()
    bi = sum(t.numel() * t.element_size() for t in host_ins)
    bo = sum(t.numel() * t.element_size() for t in dev_outs)
    return t0.elapsed_time(t1) / 1e3, bi, bo


def run_sla(args, rank, world, local):
    from gated_linear_attention_attn_b300 import sla

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    host = make_inputs(wl, seed=0)
    q, k, v, g = (t.to(dev) for t in host)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    bf16 = wl.dtype == torch.bfloat16

    # inputs within a few L2 sizes: overwrite L2 between timed steps
    scrub = L2Scrub(dev) if wl.algorithmic_bytes < 4 * L2_BYTES else None

    os.environ["SLA_FORWARD_KERNEL"] = args.forward_kernel
    blocks = wl.block_frames > 0
    cluster = sla.forward_cluster(wl.B, wl.H, wl.N, wl.rope, device=dev) \
        if bf16 and not blocks else 0
    carried = torch.zeros(wl.B, wl.H, sla.CARRIED_FLOATS, dtype=torch.float32, device=dev) \
        if blocks else None

    def step():
        if blocks:
            # one stretch of a stream: the carried state comes in and goes out in place
            sla.linattn_forward_block_causal(q, k, v, g, wl.block_tokens, out=out, rope=rope,
                                             eps=wl.eps, state_in=carried, state_out=carried,
                                             stream=stream)
        else:
            sla.linattn_forward(q, k, v, g, out=out, rope=rope, eps=wl.eps, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    status = sla.last_device_status(stream, dev)
    if status != sla.OK:
        raise RuntimeError(f"device status after warm-up: {sla.status_string(status)}")

    # -------- device-resident timing of the forward: K steps
    _barrier(world)
    torch.cuda.synchronize(dev)
    _start_sampler(dev)
    secs = _time_steps(step, args.steps, stream, scrub)
    torch.cuda.synchronize(dev)
    _barrier(world)
    secs = _max_over_ranks(secs, world, dev)
    status = sla.last_device_status(stream, dev)
    if status != sla.OK:
        raise RuntimeError(f"device status after timing: {sla.status_string(status)}")
    per_step = secs / args.steps
    value = world * wl.token_heads / per_step

    # -------- each kernel on its own, for the roofline: the fused kernel is the
    # whole forward; the two-launch plan is timed phase by phase
    kernels = {}
    plans = {}
    if blocks:
        kernels["block-causal forward (state, scan, apply)"] = {
            "us": 1e6 * per_step, "algorithmic_bytes": wl.algorithmic_bytes,
            "gbs": wl.algorithmic_bytes / per_step / 1e9}
    elif bf16 and cluster > 0:
        kernels["tc_fused_kernel"] = {"us": 1e6 * per_step,
                                      "algorithmic_bytes": wl.algorithmic_bytes,
                                      "gbs": wl.algorithmic_bytes / per_step / 1e9,
                                      "cluster": cluster}
        plans["fused"] = {"us": 1e6 * per_step, "cluster": cluster}
        with sla.forward_kernel("split"):
            for _ in range(3):
                step()
            plans["split"] = {"us": 1e6 * _time_steps(step, args.steps, stream, scrub)
                              / args.steps}
    elif bf16:
        plans["split"] = {"us": 1e6 * per_step}
    if bf16 and not blocks:
        state = sla.linattn_state(k, v, rope=rope, stream=stream)

        def k_state():
            sla.linattn_state(k, v, rope=rope, state=state, stream=stream)

        def k_apply():
            sla.linattn_apply(q, g, state, out=out, rope=rope, eps=wl.eps, stream=stream)

        per_tok = wl.d * wl.elem_size
        phases = {}
        for name, fn, unit_bytes in (("tc_state_kernel", k_state, 2 * per_tok),
                                     ("tc_apply_kernel", k_apply, 3 * per_tok)):
            for _ in range(3):
                fn()
            ksecs = _time_steps(fn, args.steps, stream, scrub) / args.steps
            alg = unit_bytes * wl.B * wl.H * wl.N
            phases[name] = {"us": 1e6 * ksecs, "algorithmic_bytes": alg,
                            "gbs": alg / ksecs / 1e9}
        if cluster > 0:
            plans["split"]["kernels"] = phases
        else:
            kernels.update(phases)
        status = sla.last_device_status(stream, dev)
        if status != sla.OK:
            raise RuntimeError(f"device status after kernel timing: {sla.status_string(status)}")

    # -------- end to end through the public call, host buffers in pinned memory
    e2e = None
    if not args.no_e2e:
        def run_e2e(ins, outs):
            if blocks:
                sla.linattn_forward_block_causal(*ins, wl.block_tokens, out=outs[0], rope=rope,
                                                 eps=wl.eps, state_in=carried,
                                                 state_out=carried, stream=stream)
            else:
                sla.linattn_forward(*ins, out=outs[0], rope=rope, eps=wl.eps, stream=stream)

        ke = max(3, min(args.steps, 10))
        _barrier(world)
        torch.cuda.synchronize(dev)
        esecs, bi, bo = pipelined_e2e(dev, stream, ke, (q, k, v, g),
                                      tuple(t.pin_memory() for t in host), (out,), run_e2e)
        esecs = _max_over_ranks(esecs, world, dev)
        _barrier(world)
        e2e = {"value": world * wl.token_heads * ke / esecs, "unit": UNIT,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": ke,
               "ms_per_step": 1e3 * esecs / ke, "note": E2E_NOTE}

    workloads = None
    if world == 1 and wl.name == HEADLINE and not args.no_workloads:
        workloads = time_workloads(args, dev, stream)

    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    if kernels:
        dom = max(kernels, key=lambda n: kernels[n]["us"])
        kd = kernels[dom]
        achieved = kd["gbs"]
        roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak,
                    "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                    if peak_src == "measured" else "fallback 6400 GB/s",
                    "algorithmic_bytes_per_launch": kd["algorithmic_bytes"],
                    "launch_us": kd["us"],
                    "traffic": stored_traffic(dom, wl.name),
                    "forward": {"achieved": wl.algorithmic_bytes / per_step / 1e9,
                                "frac": wl.algorithmic_bytes / per_step / 1e9 / peak},
                    "kernels": kernels, "plans": plans}
    else:
        achieved = wl.algorithmic_bytes / per_step / 1e9
        roofline = {"bound": "hbm", "kernel": "simt forward (both launches)",
                    "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
                    "traffic": None}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": 1e3 * per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic (seeded N(0,1) q,k,v,g on the latent token grid)",
        "config": _config(wl, world),
        "launch_plan": _forward_plan(wl, cluster),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": (3 if blocks else 1 if cluster > 0 else 2) * args.steps,
        "workloads": workloads,
        "clocks": _stop_sampler(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, host)
    print(json.dumps(line), flush=True)


BWD_METRIC = "linear-attn bwd token-heads/s; HBM GB/s as % of B300 peak"
BWD_LAUNCHES = 6
BWD_FROM_STATE_PLAN = ("backward from the forward's kept state: the same launches without "
                       "the state kernel")
BWD_PLAN = ("backward: state(k, v), apply gate terms(q, g, dout; S) + dS partials, "
            "apply masked gradient(a; S, q) -> dq + dz partials, dS merge, "
            "apply masked gradient(v; dS, k) -> dk, apply raw(k; dS) -> dv "
            "(tcgen05 state/apply kernels)")


def oracle_backward_heads(wl, tensors, heads):
    """The fp64 backward oracle on the given heads at full N; returns elapsed seconds."""
    import oracle.backward as ob   # the CPU baseline of the backward line
    import oracle.linattn as ol
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
    t0 = time.perf_counter()
    for b, h in heads:
        ang = ol.rope3d_angles(spec) if spec is not None else None
        ob.linattn_head_backward(*(x[b, h].double().numpy() for x in tensors), wl.eps, ang)
    return time.perf_counter() - t0


def run_backward(args, rank, world, local):
    """The layer's backward: dq, dk, dv, dg from q, k, v, g and the upstream gradient."""
    from gated_linear_attention_attn_b300 import sla

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    if wl.block_frames:
        raise SystemExit("the backward is timed on the bidirectional workloads")
    host = make_inputs(wl, seed=0)
    gen = torch.Generator().manual_seed(1000)
    host = host + (torch.randn(host[0].shape, generator=gen).to(wl.dtype),)
    q, k, v, g, dout = (t.to(dev) for t in host)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
    grads = tuple(torch.empty_like(q) for _ in range(4))
    stream = torch.cuda.current_stream(dev)
    alg = 9 * wl.B * wl.H * wl.N * wl.d * wl.elem_size      # 5 tensors read, 4 written
    scrub = L2Scrub(dev) if alg < 4 * L2_BYTES else None

    def step():
        sla.linattn_backward(q, k, v, g, dout, rope=rope, eps=wl.eps, grads=grads, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    if sla.last_device_status(stream, dev) != sla.OK:
        raise RuntimeError("device status after warm-up")
    _barrier(world)
    torch.cuda.synchronize(dev)
    _start_sampler(dev)
    secs = _time_steps(step, args.steps, stream, scrub)
    torch.cuda.synchronize(dev)
    _barrier(world)
    secs = _max_over_ranks(secs, world, dev)
    per_step = secs / args.steps
    # bf16: the same backward from the state a forward kept (in training the
    # forward writes each head's state and the backward reuses it)
    from_state = None
    if wl.dtype == torch.bfloat16:
        _, state = sla.linattn_forward_keep_state(q, k, v, g, rope=rope, eps=wl.eps,
                                                  stream=stream)

        def step_from_state():
            sla.linattn_backward(q, k, v, g, dout, rope=rope, eps=wl.eps, grads=grads,
                                 stream=stream, state=state)

        for _ in range(max(args.warmup, 3)):
            step_from_state()
        _barrier(world)
        torch.cuda.synchronize(dev)
        fsecs = _time_steps(step_from_state, args.steps, stream, scrub)
        torch.cuda.synchronize(dev)
        _barrier(world)
        fsecs = _max_over_ranks(fsecs, world, dev) / args.steps
        if sla.last_device_status(stream, dev) != sla.OK:
            raise RuntimeError("device status after the backward from a kept state")
        from_state = {"ms_per_step": 1e3 * fsecs, "value": world * wl.token_heads / fsecs,
                      "unit": UNIT, "hbm_frac": alg / fsecs / 1e9 / measured_peaks()[0],
                      "launch_plan": BWD_FROM_STATE_PLAN,
                      "gpu_launches_per_step": BWD_LAUNCHES - 1}
        del state
    e2e = None
    if not args.no_e2e:
        def run_e2e(ins, outs):
            sla.linattn_backward(*ins, rope=rope, eps=wl.eps, grads=outs, stream=stream)

        ke = max(3, min(args.steps, 10))
        esecs, bi, bo = pipelined_e2e(dev, stream, ke, (q, k, v, g, dout),
                                      tuple(t.pin_memory() for t in host), tuple(grads), run_e2e)
        esecs = _max_over_ranks(esecs, world, dev)
        e2e = {"value": world * wl.token_heads * ke / esecs, "unit": UNIT,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "steps": ke, "ms_per_step": 1e3 * esecs / ke, "note": E2E_NOTE}
    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    achieved = alg / per_step / 1e9
    if wl.dtype == torch.bfloat16:
        launches = BWD_LAUNCHES
        plan = BWD_PLAN
    else:
        launches = 3
        plan = "backward: state partials, query pass, key pass (fp32 FMA kernels)"
    line = {
        "metric": BWD_METRIC, "value": world * wl.token_heads / per_step, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": 1e3 * per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32",
        "data": "synthetic (seeded N(0,1) q,k,v,g and upstream gradient on the latent token grid)",
        "config": _config(wl, world),
        "launch_plan": plan,
        "roofline": {"bound": "hbm", "kernel": f"backward ({launches} launches)",
                     "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth",
                     "algorithmic_bytes_per_launch": alg, "traffic": None},
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": _stop_sampler(),
    }
    if from_state is not None:
        line["from_state"] = from_state
    if not args.no_cpu_baseline:
        heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
        done, elapsed = 0, 0.0
        while elapsed < 10.0 and done < 4 * len(heads):
            elapsed += oracle_backward_heads(wl, host, [heads[done % len(heads)]])
            done += 1
        line["cpu_baseline"] = {"value": done * wl.N / elapsed, "unit": UNIT,
                                "cores": _blas_threads(), "kind": "oracle",
                                "sample": f"{done} heads of {wl.name} at full N (fp64 numpy "
                                          f"backward, {elapsed:.1f} s)"}
    print(json.dumps(line), flush=True)


ANCHOR_METRIC = "softmax-anchor fwd token-heads/s; bf16 TFLOP/s as % of B300 peak"
FALLBACK_BF16_TFLOPS = (1800.0, 1400.0)
ANCHOR_ROWS = 256          # query rows of one head per oracle call (all N keys each)


def measured_tensor_peaks():
    """(burst, sustained) dense bf16 TFLOP/s and where they come from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            data = json.load(fh)
        return float(data["bf16_tflops"]), float(data["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return (*FALLBACK_BF16_TFLOPS, "fallback")


def oracle_anchor_rows(wl, tensors, head, rows):
    """The fp64 anchor oracle on some query rows of one head (all N keys); elapsed seconds."""
    import oracle.linattn as ol
    import oracle.softmax_anchor as oa   # the CPU baseline of the anchor line
    spec = ol.RopeSpec(*wl.grid, *wl.split, base=wl.base) if wl.rope else None
    t0 = time.perf_counter()
    oa.anchor_forward_rows(*tensors, rows, rope=spec, heads=[head])
    return time.perf_counter() - t0


def _anchor_row_sample(wl, i):
    """The i-th oracle sample: ANCHOR_ROWS consecutive query rows of one head."""
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    n = min(ANCHOR_ROWS, wl.N)
    start = (i * 7919 * n) % max(wl.N - n + 1, 1)
    return heads[i % len(heads)], list(range(start, start + n))


def anchor_cpu_baseline(wl, tensors, budget_s=10.0):
    done, elapsed, rows = 0, 0.0, 0
    while elapsed < budget_s and done < 64:
        head, sel = _anchor_row_sample(wl, done)
        elapsed += oracle_anchor_rows(wl, tensors, head, sel)
        rows += len(sel)
        done += 1
    return {"value": rows / elapsed, "unit": UNIT, "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} samples of {min(ANCHOR_ROWS, wl.N)} query rows of one head of "
                      f"{wl.name}, each against all N={wl.N} keys (fp64 numpy, "
                      f"{elapsed:.1f} s); token-heads = query rows"}


def run_anchor(args, rank, world, local):
    """The gated-softmax anchor forward: rotated q, k (RoPE pre-pass) and the attention kernel."""
    from gated_linear_attention_attn_b300 import sla

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    host = make_inputs(wl, seed=0)
    q, k, v, g = (t.to(dev) for t in host)
    rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    flops = wl.algorithmic_flops
    scrub = L2Scrub(dev) if wl.algorithmic_bytes < 4 * L2_BYTES else None

    def step():
        sla.anchor_forward(q, k, v, g, out=out, rope=rope, stream=stream)

    def attn_only():          # the same attention kernel without the RoPE pre-pass
        sla.anchor_forward(q, k, v, g, out=out, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    if sla.last_device_status(stream, dev) != sla.OK:
        raise RuntimeError("device status after warm-up")
    _barrier(world)
    torch.cuda.synchronize(dev)
    _start_sampler(dev)
    secs = _time_steps(step, args.steps, stream, scrub)
    torch.cuda.synchronize(dev)
    _barrier(world)
    secs = _max_over_ranks(secs, world, dev)
    per_step = secs / args.steps
    for _ in range(3):
        attn_only()
    attn = _time_steps(attn_only, args.steps, stream, scrub) / args.steps
    if sla.last_device_status(stream, dev) != sla.OK:
        raise RuntimeError("device status after timing")
    e2e = None
    if not args.no_e2e:
        def run_e2e(ins, outs):
            sla.anchor_forward(*ins, out=outs[0], rope=rope, stream=stream)

        ke = max(3, min(args.steps, 10))
        esecs, bi, bo = pipelined_e2e(dev, stream, ke, (q, k, v, g),
                                      tuple(t.pin_memory() for t in host), (out,), run_e2e)
        esecs = _max_over_ranks(esecs, world, dev)
        e2e = {"value": world * wl.token_heads * ke / esecs, "unit": UNIT,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "steps": ke, "ms_per_step": 1e3 * esecs / ke, "note": E2E_NOTE}
    if rank != 0:
        return
    burst, sustained, src = measured_tensor_peaks()
    achieved = flops / attn / 1e12
    line = {
        "metric": ANCHOR_METRIC, "value": world * wl.token_heads / per_step, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": 1e3 * per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q,k,v,g on the latent token grid)",
        "config": _config(wl, world),
        "launch_plan": _anchor_plan(wl),
        "note": "compute-bound: K and V of a head are re-read from L2 by every CTA",
        "roofline": {"bound": "tensor", "kernel": "anchor_attn_kernel", "achieved": achieved,
                     "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
                     "peak_source": f"{src} cuBLAS bf16, burst (bf16_tflops); the SM clock "
                                    "stays at its maximum through the timed launches",
                     "frac_of_sustained_peak": achieved / sustained,
                     "algorithmic_flops_per_launch": flops, "launch_us": 1e6 * attn,
                     "step_tflops": flops / per_step / 1e12, "traffic": None},
        "e2e": e2e,
        "gpu_launches": (2 if wl.rope else 1) * args.steps,
        "clocks": _stop_sampler(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = anchor_cpu_baseline(wl, host)
    print(json.dumps(line), flush=True)


def run_anchor_reference(args, rank, world):
    """Reference arm of an anchor workload: the fp64 oracle, ANCHOR_ROWS query rows per step."""
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    tensors = make_inputs(wl, seed=0)
    for i in range(args.warmup):
        oracle_anchor_rows(wl, tensors, *_anchor_row_sample(wl, i))
    total, rows = 0.0, 0
    for i in range(args.steps):
        head, sel = _anchor_row_sample(wl, args.warmup + i)
        total += oracle_anchor_rows(wl, tensors, head, sel)
        rows += len(sel)
    value = rows / total
    line = {
        "impl": "reference", "metric": ANCHOR_METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, world),
        "note": f"{min(ANCHOR_ROWS, wl.N)} query rows of one head (all N keys) per step on "
                "the host cores",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _blas_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} samples of {min(ANCHOR_ROWS, wl.N)} query "
                                   f"rows of {wl.name}, one per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


ATTNRES_METRIC = "AttnRes aggregation tokens/s; HBM GB/s as % of B300 peak"
ATTNRES_UNIT = "tokens/s"
ATTNRES_ROWS = 4096        # tokens per oracle call
ATTNRES_PLAN = ("attnres_kernel (bulk-copy ring of token slots, a CTA's threads over the "
                "hidden size, one barrier per token)")


def _attnres_config(wl, world):
    cfg = {"workload": wl.name, "sources": wl.H, "tokens": wl.tokens, "hidden": wl.d,
           "grid": list(wl.grid), "batch": wl.B, "input_dtype": "bfloat16", "query_dtype": "f32",
           "eps": 1e-6, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": ("inputs larger than L2 (%.0f MB vs 126 MB), steps back to back"
                  % (wl.algorithmic_bytes / 1e6) if wl.algorithmic_bytes >= 4 * L2_BYTES
                  else "L2 flushed between steps (a 252 MB buffer written, then "
                       "another read, outside the timed events)")}
    return cfg


def oracle_attnres_rows(host, rows):
    import oracle.attnres as oar   # the CPU baseline of the AttnRes line
    s, w = host
    t0 = time.perf_counter()
    oar.attnres_aggregate(s[:, rows].double().numpy(), w.double().numpy(), 1e-6)
    return time.perf_counter() - t0


def _attnres_sample(wl, i):
    n = min(ATTNRES_ROWS, wl.tokens)
    start = (i * 7919 * n) % max(wl.tokens - n + 1, 1)
    return list(range(start, start + n))


def run_attnres(args, rank, world, local):
    """The AttnRes aggregation of a later layer's input over the block summaries."""
    from gated_linear_attention_attn_b300 import sla
    from gated_linear_attention_attn_b300.workloads import make_attnres_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    wl = WORKLOADS[args.workload]
    host = make_attnres_inputs(wl, seed=0)
    s, w = (t.to(dev) for t in host)
    out = torch.empty(s.shape[1:], dtype=torch.bfloat16, device=dev)
    srcs = list(s.unbind(0))
    stream = torch.cuda.current_stream(dev)
    scrub = L2Scrub(dev) if wl.algorithmic_bytes < 4 * L2_BYTES else None

    def step():
        sla.attnres_aggregate(srcs, w, eps=1e-6, out=out, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    _barrier(world)
    torch.cuda.synchronize(dev)
    _start_sampler(dev)
    secs = _time_steps(step, args.steps, stream, scrub)
    torch.cuda.synchronize(dev)
    _barrier(world)
    secs = _max_over_ranks(secs, world, dev)
    per_step = secs / args.steps
    e2e = None
    if not args.no_e2e:
        def run_e2e(ins, outs):
            sla.attnres_aggregate(ins[0], ins[1], eps=1e-6, out=outs[0], stream=stream)

        ke = max(3, min(args.steps, 10))
        esecs, bi, bo = pipelined_e2e(dev, stream, ke, (s, w),
                                      (host[0].pin_memory(), host[1].pin_memory()), (out,),
                                      run_e2e)
        esecs = _max_over_ranks(esecs, world, dev)
        e2e = {"value": world * wl.tokens * ke / esecs, "unit": ATTNRES_UNIT,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "steps": ke, "ms_per_step": 1e3 * esecs / ke, "note": E2E_NOTE}
    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    achieved = wl.algorithmic_bytes / per_step / 1e9
    line = {
        "metric": ATTNRES_METRIC, "value": world * wl.tokens / per_step, "unit": ATTNRES_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": 1e3 * per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) summaries scaled 1+n, N(0,1)*3/sqrt(C) query)",
        "config": _attnres_config(wl, world),
        "launch_plan": ATTNRES_PLAN,
        "roofline": {"bound": "hbm", "kernel": "attnres_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth",
                     "algorithmic_bytes_per_launch": wl.algorithmic_bytes,
                     "launch_us": 1e6 * per_step,
                     "traffic": stored_traffic("attnres_kernel", wl.name)},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": _stop_sampler(),
    }
    if not args.no_cpu_baseline:
        done, elapsed, rows = 0, 0.0, 0
        while elapsed < 10.0 and done < 64:
            sel = _attnres_sample(wl, done)
            elapsed += oracle_attnres_rows(host, sel)
            rows += len(sel)
            done += 1
        line["cpu_baseline"] = {"value": rows / elapsed, "unit": ATTNRES_UNIT,
                                "cores": _blas_threads(), "kind": "oracle",
                                "sample": f"{done} samples of {min(ATTNRES_ROWS, wl.tokens)} "
                                          f"tokens of {wl.name} (fp64 numpy, {elapsed:.1f} s)"}
    print(json.dumps(line), flush=True)


def run_attnres_reference(args, rank, world):
    """Reference arm of an AttnRes workload: the fp64 oracle, ATTNRES_ROWS tokens per step."""
    if rank != 0:
        return
    from gated_linear_attention_attn_b300.workloads import make_attnres_inputs
    wl = WORKLOADS[args.workload]
    host = make_attnres_inputs(wl, seed=0)
    for i in range(args.warmup):
        oracle_attnres_rows(host, _attnres_sample(wl, i))
    total, rows = 0.0, 0
    for i in range(args.steps):
        sel = _attnres_sample(wl, args.warmup + i)
        total += oracle_attnres_rows(host, sel)
        rows += len(sel)
    value = rows / total
    line = {
        "impl": "reference", "metric": ATTNRES_METRIC, "value": value, "unit": ATTNRES_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _attnres_config(wl, world),
        "note": f"{min(ATTNRES_ROWS, wl.tokens)} tokens per step on the host cores",
        "cpu_baseline": {"value": value, "unit": ATTNRES_UNIT, "cores": _blas_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} samples of {min(ATTNRES_ROWS, wl.tokens)} "
                                   f"tokens of {wl.name}, one per step"},
        "e2e": {"value": value, "unit": ATTNRES_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------ the other configurations ----

# Timed on the headline line, each with the run's --steps and --warmup: the other
# forward configurations, the pages' 736-row 720p bucket, the block-causal form, the
# backward, and the anchor and AttnRes layers.
EXTRA_WORKLOADS = ("5b_480p", "14b_480p", "5b_720p_60s", "5b_720p_736", "5b_720p_block5",
                   "5b_720p:backward", "5b_720p:backward_from_state", "5b_720p:train_step",
                   "5b_480p:train_step", "anchor_5b_720p", "anchor_5b_480p", "attnres_5b_720p",
                   "attnres_14b_480p")


def _forward_plan(wl, cluster):
    if wl.block_frames:
        return ("block-causal: state, block scan and apply launches, %d blocks of %d tokens, "
                "carried state updated in place" % (wl.N // wl.block_tokens, wl.block_tokens))
    if wl.dtype != torch.bfloat16:
        return "fp32: state partials + apply (FMA units)"
    if cluster > 1:
        return "fused, clusters of %d CTAs per head" % cluster
    return "state + apply launches"


def _anchor_plan(wl):
    return ("RoPE pre-pass (rotated k) + anchor_attn_kernel (tcgen05, 128 queries x 128-key "
            "tiles per CTA)" if wl.rope else "anchor_attn_kernel")


def _device_inputs(wl, dev, count=4):
    """Seeded N(0, 1) inputs drawn on the device (k scaled by k_scale): the recipe's
    distribution, drawn where the timing runs; these runs are not compared with the oracle."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    out = []
    for i in range(count):
        x = torch.randn((wl.B, wl.H, wl.N, wl.d), generator=gen, device=dev, dtype=torch.float32)
        if i == 1 and wl.k_scale != 1.0:
            x.mul_(wl.k_scale)
        out.append(x.to(wl.dtype))
        del x
    return out


def time_workloads(args, dev, stream):
    """ms, throughput and roofline fraction of each EXTRA_WORKLOADS entry."""
    from gated_linear_attention_attn_b300 import sla
    peak, _ = measured_peaks()
    burst, sustained, _ = measured_tensor_peaks()
    scrub = L2Scrub(dev)

    def timed(step, alg_bytes, on=None):
        on = on if on is not None else stream
        for _ in range(max(args.warmup, 3)):
            step()
        flush = scrub if alg_bytes < 4 * L2_BYTES else None
        secs = _time_steps(step, args.steps, on, flush) / args.steps
        if sla.last_device_status(on, dev) != sla.OK:
            raise RuntimeError("device status after a workload")
        return secs, ("L2 flushed between steps" if flush else "inputs larger than L2")

    results = {}
    for entry in EXTRA_WORKLOADS:
        name, _, pass_ = entry.partition(":")
        wl = WORKLOADS[name]
        rec = {"config": _config(wl, 1)}
        if wl.layer == "attnres":
            gen = torch.Generator(device=dev)
            gen.manual_seed(0)
            src = torch.randn((wl.H, wl.tokens, wl.d), generator=gen, device=dev)
            src.mul_(torch.arange(1, wl.H + 1, device=dev, dtype=torch.float32).view(-1, 1, 1))
            src = src.to(torch.bfloat16)
            w = torch.randn((wl.d,), generator=gen, device=dev) * (3.0 / wl.d ** 0.5)
            out = torch.empty(src.shape[1:], dtype=torch.bfloat16, device=dev)
            srcs = list(src.unbind(0))
            secs, l2 = timed(lambda: sla.attnres_aggregate(srcs, w, out=out, stream=stream),
                             wl.algorithmic_bytes)
            rec.update(ms=1e3 * secs, value=wl.tokens / secs, unit=ATTNRES_UNIT,
                       hbm_gbs=wl.algorithmic_bytes / secs / 1e9,
                       hbm_frac=wl.algorithmic_bytes / secs / 1e9 / peak,
                       launch_plan=ATTNRES_PLAN, l2=l2, gpu_launches_per_step=1)
            del src, w, out, srcs
        elif wl.layer == "anchor":
            q, k, v, g = _device_inputs(wl, dev)
            rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
            out = torch.empty_like(q)
            secs, l2 = timed(lambda: sla.anchor_forward(q, k, v, g, out=out, rope=rope,
                                                        stream=stream), wl.algorithmic_bytes)
            tf = wl.algorithmic_flops / secs / 1e12
            rec.update(ms=1e3 * secs, value=wl.token_heads / secs, unit=UNIT, tflops=tf,
                       tensor_frac=tf / burst, tensor_frac_of_sustained=tf / sustained,
                       launch_plan=_anchor_plan(wl), l2=l2,
                       gpu_launches_per_step=2 if wl.rope else 1)
            del q, k, v, g, out, rope
        elif pass_ == "backward":
            q, k, v, g, dout = _device_inputs(wl, dev, 5)
            rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
            grads = tuple(torch.empty_like(q) for _ in range(4))
            alg = 9 * wl.B * wl.H * wl.N * wl.d * wl.elem_size
            secs, l2 = timed(lambda: sla.linattn_backward(q, k, v, g, dout, rope=rope,
                                                          eps=wl.eps, grads=grads,
                                                          stream=stream), alg)
            rec.update(ms=1e3 * secs, value=wl.token_heads / secs, unit=UNIT,
                       hbm_gbs=alg / secs / 1e9, hbm_frac=alg / secs / 1e9 / peak,
                       algorithmic_bytes=alg, launch_plan=BWD_PLAN, l2=l2,
                       gpu_launches_per_step=BWD_LAUNCHES)
            del q, k, v, g, dout, rope, grads
        elif pass_ in ("backward_from_state", "train_step"):
            # training: the forward keeps each head's state and the backward reuses
            # it; backward_from_state times the backward alone (the state kept by
            # one forward before the timing), train_step the forward and backward
            q, k, v, g, dout = _device_inputs(wl, dev, 5)
            rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
            grads = tuple(torch.empty_like(q) for _ in range(4))
            out = torch.empty_like(q)
            _, state = sla.linattn_forward_keep_state(q, k, v, g, out=out, rope=rope, eps=wl.eps,
                                                      stream=stream)
            cluster = sla.forward_cluster(wl.B, wl.H, wl.N, wl.rope, device=dev)
            tensor = wl.B * wl.H * wl.N * wl.d * wl.elem_size

            def bwd(on=stream):
                sla.linattn_backward(q, k, v, g, dout, rope=rope, eps=wl.eps, grads=grads,
                                     stream=on, state=state)
            on = stream
            if pass_ == "train_step":
                # The step's six or seven launches, captured as one CUDA graph and
                # replayed, as a training loop would run them: eager, the host's
                # Python and launch overhead per step (two calls) comes close to the
                # 480p step's device time and would show in it.
                def eager(s):
                    sla.linattn_forward_keep_state(q, k, v, g, out=out, rope=rope, eps=wl.eps,
                                                   state=state, stream=s)
                    bwd(s)
                on = torch.cuda.Stream(dev)
                on.wait_stream(stream)
                with torch.cuda.stream(on):
                    eager(on)                    # this stream's workspace, before the capture
                on.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=on):
                    eager(on)

                def step():
                    with torch.cuda.stream(on):
                        graph.replay()
                alg, launches = 14 * tensor, (1 if cluster > 0 else 2) + BWD_LAUNCHES - 1
                plan = (_forward_plan(wl, cluster) + ", keeping the state; then "
                        + BWD_FROM_STATE_PLAN + "; the step replayed as one CUDA graph")
            else:
                step, alg, launches = bwd, 9 * tensor, BWD_LAUNCHES - 1
                plan = BWD_FROM_STATE_PLAN
            secs, l2 = timed(step, alg, on)
            rec.update(ms=1e3 * secs, value=wl.token_heads / secs, unit=UNIT,
                       hbm_gbs=alg / secs / 1e9, hbm_frac=alg / secs / 1e9 / peak,
                       algorithmic_bytes=alg, launch_plan=plan, l2=l2,
                       gpu_launches_per_step=launches)
            del q, k, v, g, dout, rope, grads, out, state
            if pass_ == "train_step":
                del graph
        else:
            q, k, v, g = _device_inputs(wl, dev)
            rope = sla.RopeTable(wl.grid, wl.split, wl.base, device=dev) if wl.rope else None
            out = torch.empty_like(q)
            if wl.block_frames:
                carried = torch.zeros(wl.B, wl.H, sla.CARRIED_FLOATS, dtype=torch.float32,
                                      device=dev)

                def step():
                    sla.linattn_forward_block_causal(q, k, v, g, wl.block_tokens, out=out,
                                                     rope=rope, eps=wl.eps, state_in=carried,
                                                     state_out=carried, stream=stream)
                cluster, launches = 0, 3
            else:
                def step():
                    sla.linattn_forward(q, k, v, g, out=out, rope=rope, eps=wl.eps,
                                        stream=stream)
                cluster = sla.forward_cluster(wl.B, wl.H, wl.N, wl.rope, device=dev)
                launches = 1 if cluster > 0 else 2
            secs, l2 = timed(step, wl.algorithmic_bytes)
            rec.update(ms=1e3 * secs, value=wl.token_heads / secs, unit=UNIT,
                       hbm_gbs=wl.algorithmic_bytes / secs / 1e9,
                       hbm_frac=wl.algorithmic_bytes / secs / 1e9 / peak,
                       launch_plan=_forward_plan(wl, cluster), l2=l2,
                       gpu_launches_per_step=launches)
            del q, k, v, g, out, rope
        results[entry] = rec
        torch.cuda.empty_cache()
    del scrub
    torch.cuda.empty_cache()
    return results


def main():
    args = parse_args()
    rank, world, local = dist_env()
    layer = WORKLOADS[args.workload].layer
    anchor = layer == "anchor"
    if args.impl == "reference":
        if anchor:
            run_anchor_reference(args, rank, world)
        elif layer == "attnres":
            run_attnres_reference(args, rank, world)
        else:
            run_reference(args, rank, world)
        return
    if layer == "attnres":
        if args.pass_ == "backward":
            raise SystemExit("the AttnRes aggregation is timed forward only")
        run_attnres(args, rank, world, local)
    elif anchor:
        if args.pass_ == "backward":
            raise SystemExit("the anchor layer has a forward only")
        run_anchor(args, rank, world, local)
    elif args.pass_ == "backward":
        run_backward(args, rank, world, local)
    else:
        run_sla(args, rank, world, local)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
