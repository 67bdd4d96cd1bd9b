"""bench.py's JSON line on a GPU: one line with the contract's keys, run as a
separate process on small workloads (the full default line takes 155 GB and
is run by the benchmark itself)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*args):
    out = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("args", [
    ("--workload", "tiny"),                                    # full buffers, pinned-host e2e
    ("--workload", "70b_shard", "--shard-params", "8000000"),  # bucket slices, one launch
    ("--workload", "sweep_16000000_24_bf16"),                  # slices, the ring e2e
])
def test_bench_line_has_the_contract_keys(args):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _line(*args, "--steps", "5", "--warmup", "3", "--cpu-seconds", "0.5")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "gpu_launches", "clocks", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["steps"] == 5 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert d["gpu_launches"] == 5 * r["launches_per_step"] and r["launches_per_step"] >= 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"].startswith(args[1].split("_first")[0][:4])
    if "--shard-params" in args:
        assert d["e2e"] is None and r["traffic"] is None
    else:
        e = d["e2e"]
        assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0


def test_bench_clipped_line_over_bucket_slices():
    """adamw_clip on bucket slices through the stored average: norm pass, ordered
    finish, step on the average -- three launches, 2N + 34 bytes per parameter."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _line("--workload", "70b_shard", "--shard-params", "8000000", "--optimizer",
              "adamw_clip", "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    assert d["config"]["clip_path"] == "stored"
    assert d["config"]["bytes_per_param"] == 2 * 64 + 34
    assert d["roofline"]["launches_per_step"] == 3 and d["value"] > 0
    f = _line("--workload", "70b_shard", "--shard-params", "8000000", "--optimizer",
              "adamw_clip", "--clip-path", "fused", "--steps", "5", "--warmup", "3",
              "--no-cpu-baseline")
    assert f["config"]["clip_path"] == "fused"
    assert f["config"]["bytes_per_param"] == 4 * 64 + 26


def test_bench_loss_scaled_line_over_bucket_slices():
    """amp on bucket slices: fp16 gradients, the norm pass storing the average,
    the loss-scaled step on it and the scale update -- four launches."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _line("--workload", "70b_shard", "--shard-params", "8000000", "--optimizer", "amp",
              "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    assert d["config"]["clip_path"] == "stored" and "fp16" in d["config"]["workload"]
    assert d["config"]["bytes_per_param"] == 2 * 64 + 34
    assert d["roofline"]["launches_per_step"] == 4 and d["value"] > 0


@pytest.mark.parametrize("opt", ["adam", "adamw_clip", "amp"])
def test_bench_overlap_line(opt):
    """--overlap prints one line with the produce / step / serial / when-ready
    times for each optimizer form."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = _line("--overlap", "--workload", "gpt2s", "--optimizer", opt, "--bucket-elems",
              "8000000", "--steps", "3", "--warmup", "1")
    assert d["optimizer"] == opt and d["buckets"] == 4
    for k in ("ms_produce", "ms_step", "ms_produce_then_step", "ms_when_ready"):
        assert d[k] > 0, k
    assert d["ms_when_ready"] <= d["ms_produce_then_step"] * 1.05
