#!/usr/bin/env python
"""Benchmark of the fused ZeRO reduce + mixed-precision Adam step on GB300.

One step = one pass of the whole hot path over one batch of synthetic
input: the N replica gradients of this rank's shard are averaged in fixed
order, Adam updates the fp32 master/m/v, and the bf16 working copy is
written -- one call of the C ABI.

Default workload: one rank's ZeRO-3 shard of a 70B-parameter model at 64-way
data parallelism (S = 70e9/64 = 1,093,750,000 parameters, N = 64 replica
gradient slices per 4M-element bucket, 274 buckets, every bucket in one
launch).  Inputs are resident in HBM before the timed region; each step
touches 168 GB, far more than the 129 MB L2, so no flush is needed between
steps.  --workload selects the others (tiny, gpt2s, 1p3b, sweep cells).

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own
rank's shard on its own GPU, with no collective on the data path (weak
scaling); the timed region is bracketed by a barrier and a device
synchronise on every rank, and the slowest rank's time is used.

--impl reference times the CPU oracle (the plain fp64 restatement of the
method that the tests check the CUDA path against) on the host cores, on
bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "G params/s updated and achieved HBM GB/s vs ~8 TB/s roofline, at N replicas"
UNIT = "G params/s"
FALLBACK_HBM_GBS = 6800.0
# the step kernel's device code, the other replica walks and the table that
# picks the kernel for each N and gradient type: a traffic figure is void once
# any of these change
KERNEL_SOURCES = ("numerics.cuh", "kernels.cuh", "async_walk.cuh", "launch_gk.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 5 s of the workload's steps at HBM "
                         "speed, 10 to 20000)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default: 1 %% of the timed steps, 3 to 200)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="70b_shard",
                    help="tiny | gpt2s | 1p3b | 70b_shard | sweep_<S>_<N>_<bf16|fp32> "
                         "(70b_shard is the default)")
    ap.add_argument("--shard-params", type=int, default=0,
                    help="keep only the first P parameters of the workload's shard (same N, "
                         "buckets and values): a smaller case of the same kernel, for profiling")
    ap.add_argument("--bucket-launch", choices=("table", "param"), default="table",
                    help="bucket-slice workloads: 'table' -- every bucket in one launch, the "
                         "launch table written to device memory (dpopt_reduce_adam_buckets_table); "
                         "'param' -- dpopt_reduce_adam_buckets, tables in the kernel's parameter "
                         "space (2048 slice pointers per launch).  Both give the same bits.")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--overlap", action="store_true",
                    help="measure bucket-as-ready overlap: gradients produced bucket by bucket on "
                         "one stream (last bucket first), stepped on another as each is ready")
    ap.add_argument("--bucket-elems", type=int, default=0, help="override the bucket size")
    ap.add_argument("--sweep", action="store_true",
                    help="the size sweep: S in {1M, 16M, 256M, 1B} x N in {1, 2, 8, 32, 64} x "
                         "{bf16, fp32} gradients, one JSON line per cell")
    ap.add_argument("--sweep-sizes", default="", help="comma-separated S values (default all)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work budget of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=("auto", "direct", "bulk"), default="auto",
                    help="kernel policy of the library (both give identical results)")
    ap.add_argument("--optimizer", choices=("adam", "adamw_clip", "adam_allgather", "amp"),
                    default="adam",
                    help="adam: the fused reduce + Adam step; adamw_clip: the squared-norm "
                         "pre-pass then the clipped AdamW step (weight_decay 0.01, clip 1.0); "
                         "adam_allgather: the step then the ZeRO-3 all-gather of the bf16 "
                         "shard into N replica parameter buffers; amp: fp16 gradients with "
                         "dynamic loss scaling -- the unscaled squared-norm pre-pass, then the "
                         "loss-scaled, clipped AdamW step and the device-side scale update")
    ap.add_argument("--clip-path", choices=("stored", "fused"), default="stored",
                    help="adamw_clip / amp: 'stored' -- the norm pass also stores the "
                         "averaged gradient (the reduced gradient shard) and the step reads it "
                         "as one fp32 replica; 'fused' -- the step reads the N replicas again "
                         "(amp: full-buffer workloads only).  Both give the same bits.")
    ap.add_argument("--gather-path", choices=("entry", "fused", "two-pass", "separate"),
                    default="entry",
                    help="adam_allgather: 'entry' -- dpopt_reduce_adam_allgather, which runs one "
                         "kernel writing the new bf16 shard into every replica's parameter "
                         "buffer (its automatic choice: faster than the two-pass form at every "
                         "N measured); 'fused' / "
                         "'two-pass' -- the entry held to one form (dpopt_set_gather_policy); "
                         "'separate' -- the step into a separate output, then "
                         "dpopt_allgather_bf16 reads it back and broadcasts it.  All give the "
                         "same bits.")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(wl, rank: int):
    """The workload as rank `rank` runs it: the next rank's shard of the same
    model (ranks are ZeRO ranks; weak scaling, no data-path collective)."""
    from dataclasses import replace
    return replace(wl, shard_rank=(wl.shard_rank + rank) % wl.n_replicas)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's value (the only cross-rank exchange of the bench)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(world: int, shard_params: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job G params/s: every rank updates shard_params per step."""
    return world * shard_params * steps / (elapsed_ms / 1e3) / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "zero_mixed_precision_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profiles(workload: str, shard_params: int, launches_per_step: float):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None).  A summary taken on a smaller case
    of the same kernel records bytes per parameter, scaled here to the
    parameters one launch updates."""
    path = os.path.join(ROOT, "profiles", f"reduce_adam_{workload}_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != kernel_source_hash():
            return None
        if "dram_bytes_per_param" in kv:
            return float(kv["dram_bytes_per_param"]) * shard_params / max(launches_per_step, 1.0)
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.tmp = tempfile.NamedTemporaryFile(prefix="clocks_", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.tmp.close()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 7:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[3:]))
                except ValueError:
                    continue
        os.unlink(self.tmp.name)
        rows = rows[2:] if len(rows) > 4 else rows  # drop nvidia-smi's start-up samples
        if not rows:
            return None
        reasons = sorted({self.NAMES[i] for _, _, flags in rows for i, fl in enumerate(flags)
                          if fl.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_rate(wl, host_grads, budget_s: float, threads: int, max_elems: int | None = None):
    """Time the oracle on host cores over a bounded sample of the workload's shard.
    host_grads: N numpy arrays (the shard slices).  Returns (params/s, elems, calls)."""
    import numpy as np
    import oracle
    S = host_grads[0].size
    chunk = min(S, max_elems or S)
    master = np.zeros(chunk, np.float32)
    m = np.zeros(chunk, np.float32)
    v = np.zeros(chunk, np.float32)
    sl = [np.ascontiguousarray(g[:chunk]) for g in host_grads]
    done, calls, t = 0, 0, 0
    t0 = time.perf_counter()
    while True:
        t += 1
        oracle.reduce_adam_range(sl, 0, chunk, master, m, v, lr=wl.lr, beta1=wl.beta1,
                                 beta2=wl.beta2, eps=wl.eps, step=t, nthreads=threads)
        done += chunk
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return done / el, chunk, calls


def sample_elems(wl) -> int:
    """Shard elements in the oracle's timed sample: 4M, fewer at large N (the
    sample's N slices are generated on the host first)."""
    return min(4_000_000, max(250_000, 64_000_000 // wl.n_replicas))


def host_grads_for(wl, max_elems: int):
    """The rank's shard slices of step 1's gradients, generated on the host."""
    import synth
    from synth import STREAM_GRAD, stream_id
    n = min(wl.shard_elems, max_elems)
    return [synth.host_fill(wl.grad_kind, wl.shard_base, n, wl.seed, stream_id(STREAM_GRAD, r, 1),
                            wl.grad_dist(r)) for r in range(wl.n_replicas)]


def config_of(wl, kernel=None):
    return {"workload": f"{wl.name}: {wl.numel:,} params per replica buffer, N={wl.n_replicas} "
                        f"replicas, rank {wl.shard_rank} shard of {wl.shard_elems:,} params, "
                        f"{wl.bucket_elems:,}-element buckets, "
                        f"{('bf16', 'fp32', 'fp16')[wl.grad_kind]} gradients",
            "n_replicas": wl.n_replicas, "numel": wl.numel, "shard_params": wl.shard_elems,
            "bucket_elems": wl.bucket_elems,
            "bytes_per_param": wl.bytes_per_param(),
            "l2": f"inputs larger than L2: {wl.shard_elems * wl.bytes_per_param() / 1e9:.3f} GB "
                  "touched per step vs a 129 MB L2 (no flush)",
            "parallelism": "one shard per GPU, no data-path collective",
            **({"kernel_policy": kernel} if kernel else {})}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    threads = len(os.sched_getaffinity(0))
    grads = host_grads_for(wl, sample_elems(wl))
    # size one step's sample so that warmup + steps take about a minute
    rate, _, _ = oracle_rate(wl, grads, 0.5, threads, max_elems=1_000_000)
    per_step = int(max(1, min(len(grads[0]), rate * 60.0 / max(1, args.steps + args.warmup))))
    import numpy as np
    import oracle
    sl = [np.ascontiguousarray(g[:per_step]) for g in grads]
    master = np.zeros(per_step, np.float32)
    m = np.zeros(per_step, np.float32)
    v = np.zeros(per_step, np.float32)
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, nthreads=threads)
    for t in range(1, args.warmup + 1):
        oracle.reduce_adam_range(sl, 0, per_step, master, m, v, step=t, **hp)
    t0 = time.perf_counter()
    for k in range(args.steps):
        oracle.reduce_adam_range(sl, 0, per_step, master, m, v, step=args.warmup + 1 + k, **hp)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el / 1e9
    sample = (f"{per_step:,} of the {wl.shard_elems:,} shard params per step "
              f"(N={wl.n_replicas} bf16 replicas), {args.steps} steps after {args.warmup} warm-up")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded counter-based generator)", "config": config_of(wl),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import zero_mixed_precision_gb300 as dp
    from synth.device import DeviceWorkload

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    wl = rank_workload(wl, rank)
    if args.optimizer == "amp":
        if wl.layout != "full" and args.clip_path != "stored":
            raise SystemExit("amp on bucket slices runs through the stored average "
                             "(--clip-path stored)")
        wl = dataclasses.replace(wl, grad_kind=2)   # fp16 gradients, the loss-scaled recipe
    dp.dpopt_set_kernel_policy({"auto": dp.DPOPT_KERNEL_AUTO, "direct": dp.DPOPT_KERNEL_DIRECT,
                                "bulk": dp.DPOPT_KERNEL_BULK}[args.kernel])
    S, n = wl.shard_elems, wl.n_replicas
    bpp = wl.bytes_per_param()

    dev = DeviceWorkload(wl, device)
    dev.fill_states()
    dev.fill_grads(1)
    stream = torch.cuda.current_stream(device)
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)

    if args.optimizer in ("adamw_clip", "amp"):
        # one rank's view: this shard's squared norm stands in for the global one
        # (a multi-rank run adds the ranks' scalars with one all-reduce)
        sqn = torch.zeros(1, dtype=torch.float64, device=device)
        nb = 1 if wl.layout == "full" else -(-S // wl.bucket_elems)
        scratch = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, nb)[1] // 8 + 1,
                              dtype=torch.float64, device=device)
        opts = dp.step_options(weight_decay=0.01, max_grad_norm=1.0, grad_sqnorm=sqn)
    if args.optimizer == "adam_allgather":
        param_reps = [torch.empty(S * n, dtype=torch.bfloat16, device=device) for _ in range(n)]
    gather_entry = args.gather_path != "separate"
    if args.optimizer == "adam_allgather" and args.gather_path in ("fused", "two-pass"):
        pol = dp.DPOPT_GATHER_FUSED if args.gather_path == "fused" else dp.DPOPT_GATHER_SEPARATE
        if dp.dpopt_set_gather_policy(pol) != dp.DPOPT_OK:
            raise SystemExit(f"dpopt_set_gather_policy: {dp.dpopt_last_error()}")
    stored = args.clip_path == "stored"
    if args.optimizer in ("adamw_clip", "amp") and stored:
        avg = torch.empty(S, dtype=torch.float32, device=device)
    if args.optimizer == "amp":
        ls_state = torch.zeros(4, dtype=torch.int64, device=device)
        ls_cfg = dp.loss_scale_init(ls_state, init_scale=1024.0, window=1000, stream=stream)
    if wl.layout == "full":
        if args.optimizer == "adam_allgather" and gather_entry:
            def step(t):
                dp.reduce_adam_allgather(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master,
                                         dev.m, dev.v, param_reps, step=t, stream=stream, **hp)
        elif args.optimizer == "adam_allgather":
            def step(t):
                dp.reduce_adam(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m,
                               dev.v, dev.out, step=t, stream=stream, **hp)
                dp.allgather_bf16(dev.out, wl.shard_rank, param_reps, stream=stream)
        elif args.optimizer == "amp" and stored:
            def step(t):   # t is implied: the device state counts the steps taken
                dp.amp_average_sqnorm(dev.grads, wl.shard_rank, ls_state, avg, sqn, scratch,
                                      stream=stream)
                dp.amp_step([avg], 0, wl.bucket_elems, dev.master, dev.m, dev.v, dev.out,
                            weight_decay=0.01, max_grad_norm=1.0, global_sqnorm=sqn,
                            state=ls_state, cfg=ls_cfg, stream=stream, **hp)
        elif args.optimizer == "amp":
            def step(t):
                dp.amp_sqnorm(dev.grads, wl.shard_rank, ls_state, sqn, scratch, stream=stream)
                dp.amp_step(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m,
                            dev.v, dev.out, weight_decay=0.01, max_grad_norm=1.0,
                            global_sqnorm=sqn, state=ls_state, cfg=ls_cfg, stream=stream, **hp)
        elif args.optimizer == "adamw_clip" and stored:
            def step(t):
                dp.grad_average_sqnorm(dev.grads, wl.shard_rank, avg, sqn, scratch,
                                       stream=stream)
                dp.reduce_adamw([avg], 0, wl.bucket_elems, dev.master, dev.m, dev.v, dev.out,
                                step=t, opts=opts, stream=stream, **hp)
        elif args.optimizer == "adamw_clip":
            def step(t):
                dp.grad_sqnorm(dev.grads, wl.shard_rank, sqn, scratch, stream=stream)
                dp.reduce_adamw(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m,
                                dev.v, dev.out, step=t, opts=opts, stream=stream, **hp)
        else:
            def step(t):
                dp.reduce_adam(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m,
                               dev.v, dev.out, step=t, stream=stream, **hp)
    else:  # gradients delivered as per-bucket slices of the rank's shard
        if args.optimizer == "adam_allgather":
            raise SystemExit("adam_allgather runs on the full-buffer workloads")
        buckets = dev.bucket_slices()
        rows, offs = [b for _, b in buckets], [o for o, _ in buckets]
        if args.bucket_launch == "table":
            # every bucket in one launch: the launch table goes to device memory
            table = torch.empty(dp.bucket_table_bytes(n, len(rows)), dtype=torch.uint8,
                                device=device)
        else:
            table = None
        # the call's arguments marshalled once, outside the timed region
        call = dp.BucketStep(rows, offs, dev.master, dev.m, dev.v, dev.out, table)
        if args.optimizer == "amp":
            # the norm pass stores the average, unscaled by the device scale
            def step(t):   # t is implied: the device state counts the steps taken
                dp.amp_average_sqnorm_buckets(rows, offs, ls_state, avg, sqn, scratch,
                                              stream=stream)
                dp.amp_step([avg], 0, S, dev.master, dev.m, dev.v, dev.out, weight_decay=0.01,
                            max_grad_norm=1.0, global_sqnorm=sqn, state=ls_state, cfg=ls_cfg,
                            stream=stream, **hp)
        elif args.optimizer == "adamw_clip" and stored:
            # the norm pass stores the shard's average (the buckets continue one
            # another); the step reads it as one fp32 replica
            def step(t):
                dp.grad_average_sqnorm_buckets(rows, offs, avg, sqn, scratch, stream=stream)
                dp.reduce_adamw([avg], 0, S, dev.master, dev.m, dev.v, dev.out, step=t,
                                opts=opts, stream=stream, **hp)
        elif args.optimizer == "adamw_clip":
            def step(t):
                dp.grad_sqnorm_buckets(rows, offs, sqn, scratch, stream=stream)
                call.step(step=t, opts=opts, stream=stream, **hp)
        else:
            def step(t):
                call.step(step=t, stream=stream, **hp)

    def barrier():
        if world > 1:
            dist.barrier()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        uuid = str(local)
    sampler = ClockSampler(uuid)
    sampler.start()
    for t in range(1, args.warmup + 1):
        step(t)
    torch.cuda.synchronize(device)
    dp.stream_status(stream)
    time.sleep(0.3)

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(device)
    launches0 = dp.dpopt_launch_count()
    t_start.record(stream)
    for k in range(K):
        step(args.warmup + 1 + k)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    launches = dp.dpopt_launch_count() - launches0
    clocks = sampler.stop()
    dp.stream_status(stream)
    own_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(own_ms, world, device)
    # this rank's device time per step over the timed region: the step's
    # launches run back to back on one stream, so it includes the gaps between
    # them (the achieved bandwidth below is a lower bound for the kernel's own)
    kernel_ms = own_ms / K
    ms_per_step = elapsed_ms / K
    value = throughput(world, S, K, elapsed_ms)

    # end to end through the public API: host gradients in, bf16 parameters out
    esize = dev.grads[0].element_size()
    if args.optimizer != "adam" or args.shard_params:
        # (the end-to-end figure is taken for the plain fused step on whole workloads)
        return _finish(args, wl, rank, world, S, K, elapsed_ms, kernel_ms, launches, clocks,
                       None, None, stored)
    if wl.layout == "slices" and min(4, -(-S // wl.bucket_elems)) * n * wl.bucket_elems * esize \
            <= (8 << 30):
        e2e, grads = e2e_ring(args, wl, dev, stream, hp, world, barrier, K)
        return _finish(args, wl, rank, world, S, K, elapsed_ms, kernel_ms, launches, clocks,
                       e2e, grads, stored)
    if wl.layout == "slices" or n * S * esize > (8 << 30):
        # (pinned host copies of whole replica shards would not fit sensibly)
        return _finish(args, wl, rank, world, S, K, elapsed_ms, kernel_ms, launches, clocks,
                       None, None, stored)
    hs = [torch.empty(S, dtype=dev.grads[0].dtype, pin_memory=True) for _ in range(n)]
    for h, g in zip(hs, dev.shard_slices()):
        h.copy_(g)
    ds = [torch.empty(S, dtype=dev.grads[0].dtype, device=device) for _ in range(n)]
    hout = torch.empty(S, dtype=torch.bfloat16, pin_memory=True)
    Ke = max(1, min(args.e2e_steps, K))

    def timed_e2e(one_step):
        barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(Ke):
            one_step(args.warmup + K + 1 + k)
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
        dp.stream_status(stream)
        return max_over_ranks(e0.elapsed_time(e1), world, device)

    # (1) the step kernel reads the pinned host gradients in place and writes the
    # bf16 parameters into pinned host memory: each step's inputs cross the
    # host link (NVLink-C2C on a Grace-Blackwell node) inside the kernel, which
    # overlaps the inbound gradients, the arithmetic and the outbound parameters
    def in_place(t):
        dp.reduce_adam_bucket(hs, 0, dev.master, dev.m, dev.v, hout, step=t, stream=stream,
                              **hp)

    # (2) copy-engine transfers around a device-resident step, one stream
    def copies(t):
        for h, d in zip(hs, ds):
            d.copy_(h, non_blocking=True)
        dp.reduce_adam_bucket(ds, 0, dev.master, dev.m, dev.v, dev.out, step=t, stream=stream,
                              **hp)
        hout.copy_(dev.out, non_blocking=True)

    with torch.cuda.stream(stream):
        in_place(args.warmup + K + 1)          # untimed: first touch of the host pages
        ip_ms = timed_e2e(in_place)
        ce_ms = timed_e2e(copies)
    h2d, d2h = n * S * esize, S * 2
    link = host_link_h2d_gbs(device, stream)
    e2e = {"value": throughput(world, S, Ke, ip_ms), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "host_link_gbs": (h2d + d2h) * Ke / (ip_ms * 1e-3) / 1e9,
           "host_link_h2d_copy_gbs": link,
           "h2d_frac_of_copy": h2d * Ke / (ip_ms * 1e-3) / 1e9 / link,
           "path": "pinned host gradients read in place by dpopt_reduce_adam_bucket's kernel, "
                   "bf16 parameters written into pinned host memory, one launch per step",
           "copy_engine": {"value": throughput(world, S, Ke, ce_ms), "unit": UNIT,
                           "path": "pinned host gradients -> cudaMemcpyAsync -> "
                                   "dpopt_reduce_adam_bucket -> bf16 parameters back to pinned "
                                   "host, one stream"}}
    dp.stream_status(stream)
    cap = sample_elems(wl)
    grads = [(h[:cap].view(torch.int16).numpy().view("uint16") if h.dtype == torch.bfloat16
              else h[:cap].numpy()).copy() for h in hs]
    return _finish(args, wl, rank, world, S, K, elapsed_ms, kernel_ms, launches, clocks, e2e,
                   grads, stored)


def host_link_h2d_gbs(device, stream, nbytes: int = 1 << 30, reps: int = 3) -> float:
    """The host link's measured host-to-device rate: one cudaMemcpyAsync of a
    1 GB pinned buffer into device memory, timed with CUDA events (the rate
    the end-to-end figures are set against)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    src.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=device)
    with torch.cuda.stream(stream):
        dst.copy_(src, non_blocking=True)              # untimed: first touch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize(device)
    gbs = nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del src, dst
    return gbs


def e2e_ring(args, wl, dev, stream, hp, world, barrier, K):
    """End to end for bucket-slice workloads: every step, each bucket's N
    gradient slices come from pinned host memory and the new bf16 shard goes to
    pinned host memory, all inside the timed region.  The slices sit in a ring
    of R pinned host bucket slots (bucket b reads slot b mod R, so a producer
    could refill the other slots meanwhile); the one-launch bucket kernel reads
    them in place over the host link and writes the bf16 parameters straight
    to the pinned output.  The slots hold step 1's first R buckets and are not
    refilled while timed: the bytes still cross the link every step, the
    values repeat.  Returns (e2e dict, host gradient sample for the oracle)."""
    import torch

    import zero_mixed_precision_gb300 as dp
    S, n, be = wl.shard_elems, wl.n_replicas, wl.bucket_elems
    esize = dev.grads[0].element_size()
    buckets = dev.bucket_slices()
    nb = len(buckets)
    R = min(nb, 4)
    slots = []
    for k in range(R):
        ln = buckets[k][1][0].numel()
        row = [torch.empty(be, dtype=dev.grads[0].dtype, pin_memory=True) for _ in range(n)]
        for h, d in zip(row, buckets[k][1]):
            h[:ln].copy_(d)
        slots.append(row)
    hout = torch.empty(S, dtype=torch.bfloat16, pin_memory=True)
    rows = [[slots[b % R][r][:sl[0].numel()] for r in range(n)]
            for b, (_, sl) in enumerate(buckets)]
    offs = [o for o, _ in buckets]
    table = torch.empty(dp.bucket_table_bytes(n, nb), dtype=torch.uint8, device=dev.device)
    call = dp.BucketStep(rows, offs, dev.master, dev.m, dev.v, hout, table)
    h2d, d2h = n * S * esize, S * 2
    # about 3 s of timed steps at the host link's ~200 GB/s
    Ke = int(max(2, min(args.e2e_steps, K, round(3.0 / ((h2d + d2h) / 200e9)))))
    t0 = args.warmup + K + 1
    with torch.cuda.stream(stream):
        call.step(step=t0, stream=stream, **hp)   # untimed: first touch of the host pages
        torch.cuda.synchronize(dev.device)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(Ke):
            call.step(step=t0 + 1 + k, stream=stream, **hp)
        e1.record(stream)
        torch.cuda.synchronize(dev.device)
        barrier()
    dp.stream_status(stream)
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev.device)

    # The copy-engine form of the same stream: each bucket's slices copied
    # (one cudaMemcpyAsync per slice) from its pinned slot into one of two
    # device bucket slots on a copy stream, the bucket's step on the compute
    # stream behind its copies, the next bucket's copies overlapping it; the
    # bf16 shard copied back to pinned memory at the end of the step.
    dslots = [[torch.empty(be, dtype=dev.grads[0].dtype, device=dev.device) for _ in range(n)]
              for _ in range(2)]
    lens = [sl[0].numel() for _, sl in buckets]
    per_bucket = [dp.BucketStep([[x[:lens[b]] for x in dslots[b % 2]]], [offs[b]], dev.master,
                                dev.m, dev.v, dev.out) for b in range(nb)]
    cs = torch.cuda.Stream(dev.device)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def ce_step(t):
        for b in range(nb):
            k = b % 2
            cs.wait_event(free[k])        # the step two buckets back has read the slot
            with torch.cuda.stream(cs):
                for r in range(n):
                    dslots[k][r][:lens[b]].copy_(rows[b][r], non_blocking=True)
            ready[k].record(cs)
            stream.wait_event(ready[k])
            per_bucket[b].step(step=t, stream=stream, **hp)
            free[k].record(stream)
        with torch.cuda.stream(stream):
            hout.copy_(dev.out, non_blocking=True)

    t1 = t0 + Ke + 1
    ce_step(t1)                                    # untimed
    torch.cuda.synchronize(dev.device)
    barrier()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for k in range(Ke):
        ce_step(t1 + 1 + k)
    c1.record(stream)
    torch.cuda.synchronize(dev.device)
    barrier()
    dp.stream_status(stream)
    ce_ms = max_over_ranks(c0.elapsed_time(c1), world, dev.device)
    link = host_link_h2d_gbs(dev.device, stream)
    e2e = {"value": throughput(world, S, Ke, ms), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "host_link_gbs": (h2d + d2h) * Ke / (ms * 1e-3) / 1e9, "steps": Ke,
           "host_link_h2d_copy_gbs": link,
           "h2d_frac_of_copy": h2d * Ke / (ms * 1e-3) / 1e9 / link,
           "path": f"{nb} buckets x {n} gradient slices per step read in place from a ring of "
                   f"{R} pinned host bucket slots ({R * n * be * esize / 1e9:.2f} GB) by one "
                   "dpopt_reduce_adam_buckets_table launch, bf16 parameters written into pinned "
                   "host memory",
           "copy_engine": {"value": throughput(world, S, Ke, ce_ms), "unit": UNIT,
                           "host_link_gbs": (h2d + d2h) * Ke / (ce_ms * 1e-3) / 1e9,
                           "path": "each bucket's slices cudaMemcpyAsync'd (one per slice) from "
                                   "the pinned ring into two alternating device bucket slots "
                                   "on a copy stream, the bucket's step behind them, the bf16 "
                                   "shard copied back to pinned memory"}}
    # the oracle's sample: bucket 0's slices (the first elements of the shard),
    # copied out of the pinned buffers into ordinary host memory
    cap = min(be, sample_elems(wl))
    grads = [(h[:cap].view(torch.int16).numpy().view("uint16") if h.dtype == torch.bfloat16
              else h[:cap].numpy()).copy() for h in slots[0]]
    return e2e, grads


def _finish(args, wl, rank, world, S, K, elapsed_ms, kernel_ms, launches, clocks, e2e,
            host_grads, stored=False):
    import torch.distributed as dist
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    n, bpp = wl.n_replicas, wl.bytes_per_param()
    if args.optimizer in ("adamw_clip", "amp") and stored:
        # norm pass: the N replicas read, the fp32 average written (4 B); the step
        # reads that average (4 B) in place of the N replicas: g*N + 34 in all
        bpp += 8
    elif args.optimizer in ("adamw_clip", "amp"):   # the norm pre-pass reads the N gradients again
        bpp += wl.grad_bytes() * wl.n_replicas
    elif args.optimizer == "adam_allgather" and args.gather_path != "separate":
        if launches == K:
            # one fused launch per step: the bf16 copy goes to the N replica
            # buffers instead of one output (4N + 24)
            bpp += 2 * wl.n_replicas - 2
        else:
            # the step writes the own replica, the broadcast reads it and
            # writes the other N - 1 (4N + 26)
            bpp += 2 * wl.n_replicas
    elif args.optimizer == "adam_allgather":   # read the bf16 shard, write N copies (4N + 28)
        bpp += 2 + 2 * wl.n_replicas
    ms_per_step = elapsed_ms / K
    value = throughput(world, S, K, elapsed_ms)
    peak, peak_kind = load_peaks()
    achieved = S * bpp / (kernel_ms / 1e3) / 1e9
    traffic = (traffic_from_profiles(wl.name, S, launches / K)
               if args.optimizer == "adam" and not args.shard_params else None)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator, generated in HBM)",
        "config": {**config_of(wl, args.kernel), "optimizer": args.optimizer,
                   "bytes_per_param": bpp,
                   **({"clip_path": "stored" if stored else "fused"}
                      if args.optimizer in ("adamw_clip", "amp") else {}),
                   **({"gather_path": args.gather_path}
                      if args.optimizer == "adam_allgather" else {})},
        "hbm_gbs": S * bpp / (ms_per_step / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} copy bandwidth",
                     "frac_of_nominal_8tbs": achieved / 8000.0,
                     "traffic": traffic,
                     "algorithmic_bytes_per_step": S * bpp,
                     "launches_per_step": launches / K,
                     "kernel_ms_per_step": kernel_ms},
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        threads = len(os.sched_getaffinity(0))
        cap = sample_elems(wl)
        if host_grads is None:
            host_grads = host_grads_for(wl, cap)
        rate, chunk, calls = oracle_rate(wl, host_grads, args.cpu_seconds, threads,
                                         max_elems=cap)
        line["cpu_baseline"] = {
            "value": rate / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{chunk:,} of the {S:,} shard params (N={n}), {calls} Adam steps, "
                      f"{args.cpu_seconds:.0f} s of CPU work on {threads} threads"}
    if world > 1:
        dist.destroy_process_group()
    return line


def run_overlap(args, wl):
    """Bucket-as-ready against produce-then-step, on one GPU, one line of JSON:
    the plain step per bucket, or (adamw_clip, amp) the norm pass per bucket
    storing the average, then the step on the average."""
    import torch
    from dataclasses import replace

    import synth
    import zero_mixed_precision_gb300 as dp
    from synth.device import DeviceWorkload

    torch.cuda.set_device(0)
    if args.bucket_elems:
        wl = replace(wl, bucket_elems=args.bucket_elems)
    wl = replace(wl, layout="slices")
    if args.optimizer == "amp":
        wl = replace(wl, grad_kind=2)   # fp16 gradients, the loss-scaled recipe
    dev = DeviceWorkload(wl)
    dev.fill_states()
    buckets = dev.bucket_slices()
    rows, offs = [s for _, s in buckets], [o for o, _ in buckets]
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    P, C = torch.cuda.Stream(), torch.cuda.Stream()

    def produce(t, stream, events=None):
        for b in reversed(range(len(buckets))):
            off, sl = buckets[b]
            for r, x in enumerate(sl):
                synth.device_fill(x.data_ptr(), wl.grad_kind, wl.shard_base + off, x.numel(),
                                  wl.seed, synth.stream_id(synth.STREAM_GRAD, r, t),
                                  wl.grad_dist(r), stream.cuda_stream)
            if events is not None:
                events[b].record(stream)

    def timed(fn, reps):
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(P)
        C.wait_stream(P)
        for k in range(reps):
            fn(k)
        P.wait_stream(C)
        t1.record(P)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / reps

    clip = args.optimizer in ("adamw_clip", "amp")
    if args.optimizer not in ("adam", "adamw_clip", "amp"):
        raise SystemExit("--overlap measures adam, adamw_clip and amp")
    S = wl.shard_elems
    if clip:
        # the clipped (or loss-scaled) step: the norm pass storing the average,
        # then the step on it
        avg = torch.empty(S, dtype=torch.float32, device="cuda")
        sqn = torch.zeros(1, dtype=torch.float64, device="cuda")
        scratch = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, len(buckets))[1] // 8 + 1,
                              dtype=torch.float64, device="cuda")
        opts = dp.step_options(weight_decay=0.01, max_grad_norm=1.0, grad_sqnorm=sqn)
    if args.optimizer == "amp":
        ls_state = torch.zeros(4, dtype=torch.int64, device="cuda")
        ls_cfg = dp.loss_scale_init(ls_state, init_scale=1024.0, window=1000)

    def step_on_average(k, stream):
        if args.optimizer == "amp":
            dp.amp_step([avg], 0, S, dev.master, dev.m, dev.v, dev.out, weight_decay=0.01,
                        max_grad_norm=1.0, global_sqnorm=sqn, state=ls_state, cfg=ls_cfg,
                        stream=stream, **hp)
        else:
            dp.reduce_adamw([avg], 0, S, dev.master, dev.m, dev.v, dev.out, step=k + 1,
                            opts=opts, stream=stream, **hp)

    def step_batched(k, stream):
        if args.optimizer == "amp":
            dp.amp_average_sqnorm_buckets(rows, offs, ls_state, avg, sqn, scratch,
                                          stream=stream)
            step_on_average(k, stream)
        elif clip:
            dp.grad_average_sqnorm_buckets(rows, offs, avg, sqn, scratch, stream=stream)
            step_on_average(k, stream)
        else:
            dp.reduce_adam_buckets(rows, offs, dev.master, dev.m, dev.v, dev.out, step=k + 1,
                                   stream=stream, **hp)

    # each rep also runs the producer (many times the step's time): a default
    # run takes at most 200 reps
    reps = max(1, min(args.steps, 200) if getattr(args, "steps_defaulted", False) else args.steps)
    for k in range(args.warmup):
        produce(1, P)
        step_batched(k, P)
    t_prod = timed(lambda k: produce(k + 2, P), reps)
    t_step = timed(lambda k: step_batched(k, C), reps)

    def serial(k):
        produce(k + 2, P)
        step_batched(k, P)
    t_serial = timed(serial, reps)
    evs = [torch.cuda.Event() for _ in buckets]

    # buckets listed in the order they become ready (the producer goes last to first)
    rrows, roffs, revs = rows[::-1], offs[::-1], evs[::-1]

    def overlapped(k):
        produce(k + 2, P, evs)
        if args.optimizer == "amp":
            dp.amp_sqnorm_buckets_when_ready(rrows, roffs, revs, ls_state, sqn, scratch,
                                             avg_out=avg, stream=C)
            step_on_average(k, C)
        elif clip:   # the norm pass bucket by bucket; the short step on the average after
            dp.grad_sqnorm_buckets_when_ready(rrows, roffs, revs, sqn, scratch, avg_out=avg,
                                              stream=C)
            step_on_average(k, C)
        else:
            dp.reduce_adam_buckets_when_ready(rrows, roffs, revs, dev.master, dev.m, dev.v,
                                              dev.out, step=k + 1, stream=C, **hp)
        P.wait_stream(C)   # the next step's backward starts after this step's update
    t_over = timed(overlapped, reps)
    dp.stream_status(C)
    hidden = (t_serial - t_over) / t_step if t_step > 0 else 0.0
    return {"metric": "bucket-as-ready overlap of the step with gradient production",
            "optimizer": args.optimizer,
            "workload": wl.name, "n_replicas": wl.n_replicas, "shard_params": wl.shard_elems,
            "buckets": len(buckets), "bucket_elems": wl.bucket_elems, "steps": reps,
            "ms_produce": t_prod, "ms_step": t_step, "ms_produce_then_step": t_serial,
            "ms_when_ready": t_over, "fraction_of_step_hidden": hidden,
            "producer": "seeded generator kernels writing each bucket's N slices, last bucket "
                        "first, on a second stream (a stand-in for the backward pass)"}


def run_sweep(args):
    """One line per sweep cell: N slices of S elements (one bucket), one step
    per rep.  Cells whose working set is under 512 MB would sit in the 129 MB L2
    between reps, so a 1 GB buffer is written and a 256 MB one read before each
    rep and only the step is timed (flagged); cells that do not fit the free
    memory are skipped."""
    import torch

    import synth
    import zero_mixed_precision_gb300 as dp
    from synth.device import DeviceWorkload, workload_bytes

    torch.cuda.set_device(0)
    peak, peak_kind = load_peaks()
    sizes = ([int(x) for x in args.sweep_sizes.split(",")] if args.sweep_sizes
             else list(synth.SWEEP_SIZES))
    # the flush writes 1 GB, then reads 256 MB: the step starts with no line of
    # its own in L2 and no dirty line of the flush left to write back
    flush = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    clean = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    for kind in (0, 1):
        for S in sizes:
            for n in synth.SWEEP_REPLICAS:
                wl = synth.sweep_cell(S, n, kind)
                need = workload_bytes(wl)
                free, _ = torch.cuda.mem_get_info()
                line = {"cell": wl.name, "shard_params": S, "n_replicas": n,
                        "grad_dtype": "bf16" if kind == 0 else "fp32",
                        "bytes_per_param": wl.bytes_per_param()}
                if need + (4 << 30) > free:
                    line.update(skipped=f"needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free")
                    print(json.dumps(line), flush=True)
                    continue
                dev = DeviceWorkload(wl)
                dev.fill_states()
                dev.fill_grads(1)
                rows, offs = [dev.shard_slices()], [0]
                hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
                step_bytes = S * wl.bytes_per_param()
                l2_flush = step_bytes < (512 << 20)
                reps = int(min(200, max(3, 1.3e12 / max(step_bytes, 1))))
                for t in range(1, 4):
                    dp.reduce_adam_buckets(rows, offs, dev.master, dev.m, dev.v, dev.out, step=t,
                                           **hp)
                torch.cuda.synchronize()
                if l2_flush:
                    tot = 0.0
                    for k in range(reps):
                        flush.fill_(k & 0xFF)
                        clean.sum()
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record()
                        dp.reduce_adam_buckets(rows, offs, dev.master, dev.m, dev.v, dev.out,
                                               step=4 + k, **hp)
                        e1.record()
                        torch.cuda.synchronize()
                        tot += e0.elapsed_time(e1)
                    ms = tot / reps
                else:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for k in range(reps):
                        dp.reduce_adam_buckets(rows, offs, dev.master, dev.m, dev.v, dev.out,
                                               step=4 + k, **hp)
                    e1.record()
                    torch.cuda.synchronize()
                    ms = e0.elapsed_time(e1) / reps
                dp.stream_status()
                gbs = step_bytes / (ms / 1e3) / 1e9
                line.update(ms_per_step=ms, g_params_per_s=S / (ms / 1e3) / 1e9, hbm_gbs=gbs,
                            frac_of_measured=gbs / peak, frac_of_8tbs=gbs / 8000.0,
                            peak_source=peak_kind, reps=reps,
                            l2="flushed before each rep (1 GB written, 256 MB read), step "
                               "timed alone: not a roofline figure" if l2_flush
                               else "working set above L2")
                print(json.dumps(line), flush=True)
                del dev, rows, offs
                torch.cuda.empty_cache()


def resolve_workload(name: str):
    """A named workload, one sweep cell written sweep_<S>_<N>_<bf16|fp32>, or
    full_<S>_<N>_<bf16|fp32>: the sweep cell's values as N full replica buffers
    of S*N elements, rank 0's shard (the layout the all-gather runs on)."""
    import synth
    if name in synth.WORKLOADS:
        return synth.WORKLOADS[name]
    parts = name.split("_")
    if len(parts) == 4 and parts[0] in ("sweep", "full") and parts[3] in ("bf16", "fp32"):
        wl = synth.sweep_cell(int(parts[1]), int(parts[2]), 0 if parts[3] == "bf16" else 1)
        if parts[0] == "full":
            wl = dataclasses.replace(wl, name="full" + wl.name[len("sweep"):], layout="full")
        return wl
    raise SystemExit(f"unknown workload {name}")


def default_steps(wl) -> int:
    """Timed steps when none are given: about 5 s of steps at 6.5 TB/s."""
    est_s = wl.shard_elems * (wl.grad_bytes() * wl.n_replicas + 26) / 6.5e12
    return int(max(10, min(20000, round(5.0 / max(est_s, 1e-9)))))


def main(argv=None):
    args = parse_args(argv)
    import synth
    wl = resolve_workload(args.workload)
    if args.shard_params:
        if not 0 < args.shard_params <= wl.shard_elems:
            raise SystemExit(f"--shard-params must lie in [1, {wl.shard_elems}]")
        wl = dataclasses.replace(wl, numel=args.shard_params * wl.n_replicas, shard_rank=0,
                                 name=f"{wl.name}_first{args.shard_params}")
    args.steps_defaulted = args.steps is None
    if args.steps is None:
        args.steps = default_steps(wl)
    if args.warmup is None:
        args.warmup = max(3, min(200, args.steps // 100))
    if args.overlap:
        print(json.dumps(run_overlap(args, wl)), flush=True)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        line = run_reference(args, wl)
    else:
        line = run_ours(args, wl)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
