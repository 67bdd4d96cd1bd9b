"""The one-launch bucket entry (dpopt_reduce_adam_buckets_table): every bucket
in one kernel launch, the launch table written to caller-owned device memory.

Its results must be bitwise those of the parameter-space entry
(dpopt_reduce_adam_buckets / dpopt_reduce_adamw_buckets), which needs several
launches once a call has more than 2048 slice pointers, and match the oracle
step by step.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity
from tests.test_gpu_parity import HP, _small_workload, f32, to_dev_grad, u16

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
else:
    dp = None


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _slices(wl, t, bucket, shift=0):
    """Bucket slices of step t's gradients, each slice its own allocation
    starting `shift` elements into it (shift != 0: unaligned slices)."""
    S = wl.shard_elems
    rows, offs = [], []
    host = [parity.grad_host_range(wl, r, t, wl.shard_base, S) for r in range(wl.n_replicas)]
    for off in range(0, S, bucket):
        ln = min(bucket, S - off)
        row = []
        for r in range(wl.n_replicas):
            big = torch.zeros(ln + 8, dtype={0: torch.bfloat16, 1: torch.float32,
                                             2: torch.float16}[wl.grad_kind], device="cuda")
            big[shift:shift + ln] = to_dev_grad(host[r][off:off + ln])
            row.append(big[shift:shift + ln])
        rows.append(row)
        offs.append(off)
    return rows, offs


def _run(wl, bucket, entry, steps=(1, 2), shift=0, opts_fn=None, check=False):
    S = wl.shard_elems
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
    out = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    nb = -(-S // bucket)
    table = torch.empty(dp.bucket_table_bytes(wl.n_replicas, nb) + 64, dtype=torch.uint8,
                        device="cuda")
    launches = []
    for t in steps:
        prev = [f32(x) for x in st]
        rows, offs = _slices(wl, t, bucket, shift)
        opts = opts_fn(t) if opts_fn else None
        c0 = dp.dpopt_launch_count()
        if entry == "table":
            dp.reduce_adam_buckets_table(rows, offs, *st, out, table, step=t, opts=opts, **HP)
        elif opts is not None:
            dp.reduce_adamw_buckets(rows, offs, *st, out, step=t, opts=opts, **HP)
        else:
            dp.reduce_adam_buckets(rows, offs, *st, out, step=t, **HP)
        launches.append(dp.dpopt_launch_count() - c0)
        dp.stream_status()
        if check:
            parity.check_step(wl, np.arange(S), t, prev, [f32(x) for x in st] + [u16(out)],
                              f"table N={wl.n_replicas} S={S} shift={shift}")
    return [f32(x) for x in st] + [u16(out)], launches


@pytest.mark.parametrize("n,S,bucket,kind", [
    (64, 40_003, 997, 0),     # 41 buckets x 64 = 2624 pointers: two parameter-space launches
    (64, 70_000, 1_000, 1),   # fp32, 70 buckets
    (13, 300_007, 1_999, 0),  # 151 buckets: beyond 128 segments per launch
    (24, 60_001, 401, 0),     # 150 buckets: the shared-memory replica walk over the table
    (40, 20_000, 100, 2),     # fp16, 200 buckets, the same walk
    (4, 100_000, 333, 2),     # fp16, 301 buckets
    (2, 8_192, 4_096, 0),     # two whole buckets, 32-byte state accesses
    (1, 5_000, 7, 0),         # 715 tiny buckets, scalar tails everywhere
])
def test_table_entry_is_bitwise_the_parameter_space_entry(n, S, bucket, kind):
    _need_gpu()
    wl = _small_workload(n, S, kind=kind)
    a, la = _run(wl, bucket, "table", check=True)
    b, lb = _run(wl, bucket, "param")
    assert la == [1, 1]
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("shift", [1, 4])
def test_table_entry_unaligned_slices(shift):
    _need_gpu()
    wl = _small_workload(64, 9_001, kind=0)
    a, _ = _run(wl, 1_000, "table", shift=shift, check=True)
    b, _ = _run(wl, 1_000, "param", shift=shift)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_table_entry_with_adamw_and_clipping():
    _need_gpu()
    wl = _small_workload(16, 50_000, kind=0, rank=0)
    S = wl.shard_elems
    sq = torch.empty(1, dtype=torch.float64, device="cuda")

    def opts_fn(t):
        # the squared norm of this shard's averaged gradient, from the oracle
        host = [parity.grad_host_range(wl, r, t, wl.shard_base, S) for r in range(wl.n_replicas)]
        sq.fill_(oracle.grad_sqnorm(host, 0, S, 1.0))
        return dp.step_options(weight_decay=0.01, max_grad_norm=1e-4, grad_sqnorm=sq)
    a, la = _run(wl, 3_001, "table", opts_fn=opts_fn)
    b, _ = _run(wl, 3_001, "param", opts_fn=opts_fn)
    assert la == [1, 1]
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_table_entry_reads_host_slices_in_place():
    """Pinned host slices (the benchmark's end-to-end ring) give the bits of
    device slices."""
    _need_gpu()
    wl = _small_workload(8, 30_000, kind=0)
    S, bucket = wl.shard_elems, 4_000
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    res = []
    for where in ("device", "host"):
        st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        out = (torch.empty(S, dtype=torch.bfloat16, device="cuda") if where == "device"
               else torch.empty(S, dtype=torch.bfloat16, pin_memory=True))
        rows, offs = _slices(wl, 1, bucket)
        if where == "host":
            rows = [[x.cpu().pin_memory() for x in row] for row in rows]
        table = torch.empty(dp.bucket_table_bytes(wl.n_replicas, len(rows)), dtype=torch.uint8,
                            device="cuda")
        dp.reduce_adam_buckets_table(rows, offs, *st, out, table, step=1, **HP)
        dp.stream_status()
        torch.cuda.synchronize()
        res.append([f32(x) for x in st] + [u16(out)])
    for x, y in zip(*res):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_table_entry_rejects_a_small_table_without_launching():
    _need_gpu()
    wl = _small_workload(4, 4_000, kind=0)
    rows, offs = _slices(wl, 1, 1_000)
    st = [torch.zeros(wl.shard_elems, device="cuda") for _ in range(3)]
    out = torch.empty(wl.shard_elems, dtype=torch.bfloat16, device="cuda")
    table = torch.empty(dp.bucket_table_bytes(4, 4) - 8, dtype=torch.uint8, device="cuda")
    c0 = dp.dpopt_launch_count()
    with pytest.raises(dp.DpoptError):
        dp.reduce_adam_buckets_table(rows, offs, *st, out, table, step=1, **HP)
    assert dp.dpopt_launch_count() == c0
    assert not st[0].any()


def test_contiguous_buckets_are_joined_into_one_launch():
    """Buckets that are consecutive views of flat replica buffers (contiguous
    gradients) are joined into one segment: one launch from the parameter-space
    entry, with the bits of the same buckets held in separate allocations."""
    _need_gpu()
    wl = _small_workload(64, 300_000, kind=0)
    S, bucket = wl.shard_elems, 1_000
    host = [parity.grad_host_range(wl, r, 1, wl.shard_base, S) for r in range(wl.n_replicas)]
    flat = [to_dev_grad(h) for h in host]
    rows = [[g[off:off + min(bucket, S - off)] for g in flat] for off in range(0, S, bucket)]
    offs = list(range(0, S, bucket))
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    res = []
    for entry in ("joined", "separate"):
        st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        out = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        c0 = dp.dpopt_launch_count()
        if entry == "joined":
            dp.reduce_adam_buckets(rows, offs, *st, out, step=1, **HP)
            assert dp.dpopt_launch_count() - c0 == 1
        else:
            sep, _ = _slices(wl, 1, bucket)
            table = torch.empty(dp.bucket_table_bytes(wl.n_replicas, len(sep)),
                                dtype=torch.uint8, device="cuda")
            dp.reduce_adam_buckets_table(sep, offs, *st, out, table, step=1, **HP)
        dp.stream_status()
        res.append([f32(x) for x in st] + [u16(out)])
    for x, y in zip(*res):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
