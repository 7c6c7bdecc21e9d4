"""The reference arm of bench.py (the fp64 oracle on the host cores) keeps the
JSON-line contract for every layer it can time: one line with impl, metric,
value, unit, the step counts, a cpu_baseline describing the run and an e2e
object with no host-device traffic.  Runs on the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(workload):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", workload, "--steps", "1", "--warmup", "0"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload,unit", [("tiny_fp32", "token-heads/s"),
                                           ("anchor_5b_480p", "token-heads/s"),
                                           ("attnres_14b_480p", "tokens/s")])
def test_reference_arm_line(workload, unit):
    line = _reference_line(workload)
    assert line["impl"] == "reference"
    assert line["unit"] == unit and line["value"] > 0
    assert line["steps"] == 1 and line["warmup"] == 0 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["gpu_launches"] == 0
    assert line["config"]["workload"] == workload
    # the config names the workload only: no run notes or launch plans in it, so both
    # arms of a workload carry the same config
    assert "note" not in line["config"] and "launch_plan" not in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == unit
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_headline_line_times_known_workloads_and_passes():
    """Every entry the headline line times beside the headline names a workload of
    the table and a pass bench.py knows how to time (forward, backward, the backward
    from a kept state, the training step); the training passes are on bf16 workloads
    of the bidirectional layer."""
    sys.path.insert(0, ROOT)
    import bench
    from gated_linear_attention_attn_b300.workloads import WORKLOADS
    passes = {"", "backward", "backward_from_state", "train_step"}
    for entry in bench.EXTRA_WORKLOADS:
        name, _, pass_ = entry.partition(":")
        assert name in WORKLOADS, entry
        assert pass_ in passes, entry
        if pass_:
            wl = WORKLOADS[name]
            assert wl.layer == "linear" and not wl.block_frames, entry
            assert str(wl.dtype) == "torch.bfloat16", entry
    assert len(set(bench.EXTRA_WORKLOADS)) == len(bench.EXTRA_WORKLOADS)
