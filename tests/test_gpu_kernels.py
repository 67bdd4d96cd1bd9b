"""The two kernels of the library -- direct loads and bulk-copy (TMA) staging --
give bitwise identical results, agree with the oracle, and report a bounded
device-side wait that runs out without losing the CUDA context."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from tests import parity
from tests.parity import oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import _run_small_full, _small_workload, f32, u16
else:
    dp = None


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _both(wl, **kw):
    with dp.kernel_policy(dp.DPOPT_KERNEL_DIRECT):
        a = _run_small_full(wl, **kw)
    with dp.kernel_policy(dp.DPOPT_KERNEL_BULK):
        b = _run_small_full(wl, **kw)
    return a, b


@pytest.mark.parametrize("n,kind", [(1, 0), (2, 0), (3, 0), (4, 0), (6, 0), (8, 0), (13, 0),
                                    (1, 1), (3, 1), (4, 1)])
@pytest.mark.parametrize("S", [7, 8, 2047, 2048, 2049, 100_003])
def test_bulk_copy_kernel_is_bitwise_equal_to_direct(n, kind, S):
    """Where the ring fits (bf16 N <= 6, fp32 N <= 3) the bulk-copy kernel runs;
    beyond it the bulk policy falls back to direct loads: same bits either way."""
    _need_gpu()
    wl = _small_workload(n, S, kind=kind)
    a, b = _both(wl, steps=(1, 2))
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    parity.check(refs[-1], *b, where=f"bulk N={n} S={S}")


@pytest.mark.parametrize("n,kind", [(2, 1), (3, 1), (5, 0), (6, 0)])
def test_bulk_copy_kernel_batched_buckets(n, kind):
    _need_gpu()
    wl = _small_workload(n, 123_457, kind=kind, rank=1)
    for bucket in (2048, 4099, 10_000):
        a, b = _both(wl, entry="buckets", bucket=bucket, steps=(1, 2))
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), bucket


def test_bulk_policy_falls_back_where_it_cannot_apply():
    """Unaligned buffers and replica counts beyond the shared-memory ring still
    run (through the direct-load kernel) under the bulk policy."""
    _need_gpu()
    wl = _small_workload(32, 9_000)
    a, b = _both(wl, steps=(1,))
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_bulk_copy_kernel_on_the_gpt2s_workload_matches_direct():
    _need_gpu()
    from synth.device import DeviceWorkload
    wl = synth.WORKLOADS["gpt2s"]
    outs = []
    for pol in (dp.DPOPT_KERNEL_DIRECT, dp.DPOPT_KERNEL_BULK):
        dev = DeviceWorkload(wl)
        dev.fill_states()
        with dp.kernel_policy(pol):
            for t in (1, 2):
                dev.fill_grads(t)
                dp.reduce_adam(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m, dev.v,
                               dev.out, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=t)
        dp.stream_status()
        outs.append([dev.master.clone(), dev.m.clone(), dev.v.clone(), dev.out.clone()])
        del dev
    for x, y in zip(*outs):
        assert torch.equal(x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32),
                           y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32))
    torch.cuda.empty_cache()


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    _need_gpu()
    stream = torch.cuda.current_stream().cuda_stream
    assert dp.dpopt_stream_status(stream) == dp.DPOPT_OK
    # about a millisecond at GB300 clocks: nothing ever arrives on the barrier
    assert dp.dpopt_selftest_wait_timeout(2_000_000, stream) == dp.DPOPT_OK
    assert dp.dpopt_stream_status(stream) == dp.DPOPT_ERR_TIMEOUT
    # the status word is cleared by the read, and the device still computes
    assert dp.dpopt_stream_status(stream) == dp.DPOPT_OK
    wl = _small_workload(4, 4096)
    got = _run_small_full(wl, steps=(1,))
    refs = oracle_trajectory(wl, np.arange(4096), 1, 1)
    parity.check(refs[0], *got, where="after time-out")
