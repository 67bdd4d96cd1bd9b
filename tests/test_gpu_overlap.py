"""Bucket-as-ready: buckets produced on one stream (a stand-in backward pass,
last bucket first) are stepped on another as each one's event fires; the
result equals the batched step bit for bit and matches the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from synth.device import DeviceWorkload
from tests import parity
from tests.parity import oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import f32, u16
else:
    dp = None


def _wl():
    return synth.Workload(name="overlap", n_replicas=4, numel=4 * 3_000_001, shard_rank=2,
                          bucket_elems=400_000, seed=51, grad_dist=lambda r: synth.Dist(0.0, 1e-3),
                          master_dist=synth.Dist(0.0, 0.02), m_dist=None, v_dist=None, steps=2,
                          layout="slices")


def _produce(dev, wl, t, stream, events):
    """Fill step t's gradients bucket by bucket, last bucket first, recording
    each bucket's event on `stream` when its N slices are written."""
    buckets = dev.bucket_slices()
    for b in reversed(range(len(buckets))):
        off, sl = buckets[b]
        for r, x in enumerate(sl):
            synth.device_fill(x.data_ptr(), wl.grad_kind, wl.shard_base + off, x.numel(), wl.seed,
                              synth.stream_id(synth.STREAM_GRAD, r, t), wl.grad_dist(r),
                              stream.cuda_stream)
        events[b].record(stream)
    return buckets


def test_when_ready_equals_the_batched_step_and_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _wl()
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    results = []
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, wl.shard_elems, 20_000),
                                    np.arange(wl.shard_elems - 100, wl.shard_elems)]))
    for mode in ("ready", "batched"):
        dev = DeviceWorkload(wl)
        dev.fill_states()
        torch.cuda.synchronize()
        for t in (1, 2):
            prev = [f32(x)[idx] for x in (dev.master, dev.m, dev.v)]
            nb = -(-wl.shard_elems // wl.bucket_elems)
            events = [torch.cuda.Event() for _ in range(nb)]
            buckets = _produce(dev, wl, t, producer, events)
            rows, offs = [s for _, s in buckets], [o for o, _ in buckets]
            if mode == "ready":   # in readiness order: last bucket first
                dp.reduce_adam_buckets_when_ready(rows[::-1], offs[::-1], events[::-1],
                                                  dev.master, dev.m, dev.v, dev.out, step=t,
                                                  stream=consumer, **hp)
            else:
                consumer.wait_stream(producer)
                dp.reduce_adam_buckets(rows, offs, dev.master, dev.m, dev.v, dev.out, step=t,
                                       stream=consumer, **hp)
            consumer.synchronize()
            dp.stream_status(consumer)
            if mode == "ready":
                got = [f32(x)[idx] for x in (dev.master, dev.m, dev.v)] + [u16(dev.out)[idx]]
                parity.check_step(wl, idx, t, prev, got, "when_ready")
        results.append([f32(dev.master), f32(dev.m), f32(dev.v), u16(dev.out)])
    for a, b in zip(*results):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    refs = oracle_trajectory(wl, idx, 1, 2)
    parity.check(refs[-1], *(x[idx] for x in results[0]), where="when_ready")


def test_null_events_mean_ready_now():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _wl()
    dev = DeviceWorkload(wl)
    dev.fill_states()
    dev.fill_grads(1)
    buckets = dev.bucket_slices()
    rows, offs = [s for _, s in buckets], [o for o, _ in buckets]
    dp.reduce_adam_buckets_when_ready(rows, offs, [None] * len(rows), dev.master, dev.m, dev.v,
                                      dev.out, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2,
                                      eps=wl.eps, step=1)
    dp.stream_status()
    refs = oracle_trajectory(wl, np.arange(0, wl.shard_elems, 997), 1, 1)
    parity.check(refs[0], f32(dev.master)[::997], f32(dev.m)[::997], f32(dev.v)[::997],
                 u16(dev.out)[::997], where="null events")


def test_norm_pass_when_ready_then_the_step_on_the_average():
    """The clipping pre-pass bucket by bucket behind the producer's events,
    storing the average; then the clipped step reads the average.  The norm is
    bitwise that of the batched norm over the same buckets held apart, the
    average that of the joined buckets, the states those of the fused bucket
    step, and the norm within the oracle's bound."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from tests.parity import grad_host_range
    wl = _wl()
    S, n = wl.shard_elems, wl.n_replicas
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    dev = DeviceWorkload(wl)
    dev.fill_states()
    nb = -(-S // wl.bucket_elems)

    def scratch():
        return torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, nb)[1] // 8 + 1,
                           dtype=torch.float64, device="cuda")
    events = [torch.cuda.Event() for _ in range(nb)]
    torch.cuda.synchronize()
    buckets = _produce(dev, wl, 1, producer, events)
    rows, offs = [s for _, s in buckets], [o for o, _ in buckets]
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    avg = torch.full((S,), float("nan"), device="cuda")
    c0 = dp.dpopt_launch_count()
    dp.grad_sqnorm_buckets_when_ready(rows[::-1], offs[::-1], events[::-1], sq, scratch(),
                                      avg_out=avg, stream=consumer)
    assert dp.dpopt_launch_count() - c0 == nb + 1      # one pass per bucket, one finish
    consumer.synchronize()
    dp.stream_status(consumer)
    # the same buckets held apart (no joining), batched; and joined, storing the average
    apart = [[x.clone() for x in row] for row in rows]
    sq_apart = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_sqnorm_buckets(apart, offs, sq_apart, scratch())
    sq_joined = torch.zeros(1, dtype=torch.float64, device="cuda")
    avg_joined = torch.full((S,), float("nan"), device="cuda")
    dp.grad_average_sqnorm_buckets(rows, offs, avg_joined, sq_joined, scratch())
    dp.stream_status()
    assert torch.equal(sq, sq_apart)
    assert np.array_equal(f32(avg).view(np.uint32), f32(avg_joined).view(np.uint32))
    gh = [grad_host_range(wl, r, 1, wl.shard_base, S) for r in range(n)]
    want = oracle.grad_sqnorm(gh, 0, S, 1.0)
    assert float(sq.item()) == pytest.approx(want, rel=4 * S * 2.0 ** -53)
    # the clipped step on the average, against the fused bucket step with the same norm
    max_norm = 0.3 * float(np.sqrt(want))
    res = []
    for form in ("average", "fused"):
        st = [x.clone() for x in (dev.master, dev.m, dev.v)]
        out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        opts = dp.step_options(weight_decay=0.01, max_grad_norm=max_norm, grad_sqnorm=sq)
        if form == "average":
            dp.reduce_adamw([avg], 0, S, *st, out, step=1, opts=opts, **hp)
        else:
            dp.reduce_adamw_buckets(rows, offs, *st, out, step=1, opts=opts, **hp)
        dp.stream_status()
        res.append([f32(x) for x in st] + [u16(out)])
    for a, b in zip(*res):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    idx = np.arange(0, S, 101)
    c = oracle.grad_scale(want, max_norm, 1.0)
    base = wl.shard_base
    parity.check_step(wl, idx, 1, [f32(x)[idx] for x in (dev.master, dev.m, dev.v)],
                      [x[idx] for x in res[0]], "norm when ready, step on the average",
                      grads_fn=lambda r, _t: gh[r][idx], weight_decay=0.01,
                      gscale_fn=lambda _t, _g: c)


def test_loss_scaled_norm_when_ready_equals_the_batched_run():
    """Five loss-scaled iterations, fp16 gradients produced bucket by bucket
    (an Inf planted at iteration 3): the norm pass behind each bucket's event
    then the step on the stored average skips, rescales and steps exactly as
    the batched run over joined buckets (no clipping: only the overflow test
    reads the norm, so the two partitions give the same decisions and bits)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dataclasses import replace
    wl = replace(_wl(), grad_kind=2, numel=4 * 1_000_003, bucket_elems=150_000)
    S = wl.shard_elems
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    nb = -(-S // wl.bucket_elems)
    res = []
    for mode in ("ready", "batched"):
        dev = DeviceWorkload(wl)
        dev.fill_states()
        state = torch.zeros(4, dtype=torch.int64, device="cuda")
        cfg = dp.loss_scale_init(state, init_scale=1024.0, window=2, hysteresis=1,
                                 min_scale=1.0)
        avg = torch.empty(S, device="cuda")
        sq = torch.zeros(1, dtype=torch.float64, device="cuda")
        scratch = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, nb)[1] // 8 + 1,
                              dtype=torch.float64, device="cuda")
        trail = []
        torch.cuda.synchronize()
        for t in range(1, 6):
            events = [torch.cuda.Event() for _ in range(nb)]
            buckets = _produce(dev, wl, t, producer, events)
            rows, offs = [s for _, s in buckets], [o for o, _ in buckets]
            if t == 3:   # an overflow in one replica of the middle bucket
                with torch.cuda.stream(producer):
                    rows[nb // 2][1][7] = float("inf")
                events[nb // 2].record(producer)
            if mode == "ready":
                dp.amp_sqnorm_buckets_when_ready(rows[::-1], offs[::-1], events[::-1], state, sq,
                                                 scratch, avg_out=avg, stream=consumer)
            else:
                consumer.wait_stream(producer)
                dp.amp_average_sqnorm_buckets(rows, offs, state, avg, sq, scratch,
                                              stream=consumer)
            dp.amp_step([avg], 0, S, dev.master, dev.m, dev.v, dev.out, weight_decay=0.01,
                        max_grad_norm=0.0, global_sqnorm=sq, state=state, cfg=cfg,
                        stream=consumer, **hp)
            producer.wait_stream(consumer)
            consumer.synchronize()
            dp.stream_status(consumer)
            st = dp.read_loss_scale(state)
            trail.append((st.scale, st.step, st.skipped, st.last_overflow))
        res.append((trail, [f32(dev.master), f32(dev.m), f32(dev.v), u16(dev.out)]))
    assert res[0][0] == res[1][0]
    assert res[0][0][2][3] == 1 and res[0][0][-1][2] == 1      # iteration 3 skipped
    for a, b in zip(res[0][1], res[1][1]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
