"""Host logic of the multi-rank benchmark, on CPU with gloo, world size 2:
each rank takes its own shard, only the timing is exchanged (max over ranks),
and only rank 0 prints."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = bench.rank_workload(synth.WORKLOADS["gpt2s"], rank)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    q.put((rank, wl.shard_rank, wl.shard_base, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_ranks_take_distinct_shards_and_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, b0, t0), (r1, s1, b1, t1) = res
    assert (s0, s1) == (0, 1) and b1 == 31_000_000 and b0 == 0
    assert t0 == t1 == 15.0


def test_throughput_is_the_whole_job_aggregate():
    import bench
    assert bench.throughput(2, 31_000_000, 100, 1000.0) == pytest.approx(6.2)
    assert bench.throughput(1, 31_000_000, 100, 1000.0) == pytest.approx(3.1)


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "3", "--warmup", "1"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "G params/s"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_default_timed_steps_are_about_five_seconds_of_the_workload():
    """Without --steps the timed region is sized to the workload: about 5 s at
    6.5 TB/s, between 10 and 20000 steps, so that every workload's default run
    ends within minutes (70b_shard moves 168 GB per step)."""
    sys.path.insert(0, ROOT)
    import bench
    for name in ("tiny", "gpt2s", "1p3b", "70b_shard", "sweep_1000000000_64_fp32"):
        wl = bench.resolve_workload(name)
        k = bench.default_steps(wl)
        assert 10 <= k <= 20000
        per_step_s = wl.shard_elems * (wl.grad_bytes() * wl.n_replicas + 26) / 6.5e12
        assert k == 20000 or abs(k * per_step_s - 5.0) < per_step_s + 1e-9
    assert bench.default_steps(bench.resolve_workload("gpt2s")) == 20000
    assert bench.default_steps(bench.resolve_workload("70b_shard")) == 193


def test_default_workload_and_named_layouts():
    """The default line is the 70B model's 1/64 shard; sweep_ names give bucket
    slices, full_ names the same cell as N full replica buffers; --shard-params
    keeps the first P parameters of the same workload."""
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args([])
    assert args.workload == "70b_shard" and args.bucket_launch == "table"
    wl = bench.resolve_workload("70b_shard")
    assert (wl.n_replicas, wl.shard_elems, wl.bucket_elems) == (64, 1_093_750_000, 4_000_000)
    s = bench.resolve_workload("sweep_256000000_24_bf16")
    f = bench.resolve_workload("full_256000000_24_fp32")
    assert s.layout == "slices" and f.layout == "full"
    assert (f.shard_elems, f.n_replicas, f.grad_kind) == (256_000_000, 24, 1)
    assert f.name.startswith("full_")
    with pytest.raises(SystemExit):
        bench.resolve_workload("sweep_1_2_int8")
    assert bench.sample_elems(wl) == 1_000_000 and bench.sample_elems(s) == 2_666_666
    assert bench.sample_elems(bench.resolve_workload("gpt2s")) == 4_000_000


def test_traffic_is_scaled_per_parameter_and_void_on_other_sources(tmp_path, monkeypatch):
    """A traffic summary taken on a smaller case records bytes per parameter,
    scaled to the parameters of one launch; a summary taken on other kernel
    sources gives no figure."""
    sys.path.insert(0, ROOT)
    import bench
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "reduce_adam_w_traffic.txt").write_text(
        "# comment: ignored\ndram_bytes_per_param: 150.5\nsource_sha256: abc\n")
    (tmp_path / "profiles" / "reduce_adam_v_traffic.txt").write_text(
        "dram_bytes_per_launch: 1000\nsource_sha256: abc\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    assert bench.traffic_from_profiles("w", 1_000_000, 1.0) == pytest.approx(150.5e6)
    assert bench.traffic_from_profiles("w", 1_000_000, 2.0) == pytest.approx(75.25e6)
    assert bench.traffic_from_profiles("v", 123, 1.0) == 1000.0
    assert bench.traffic_from_profiles("missing", 1, 1.0) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "other")
    assert bench.traffic_from_profiles("w", 1_000_000, 1.0) is None
