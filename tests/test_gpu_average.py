"""The stored averaged gradient (the reduced gradient shard of ZeRO stage 2) on
the GPU: the average the norm pass writes agrees with the oracle's fixed-order
average, and the two-pass path -- norm pass storing the average, then the step
reading it as one fp32 replica -- gives bit for bit the states of the fused
path that reads the N replicas in the step, for clipped AdamW and for the
loss-scaled fp16 step (overflow skips included)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests.parity import grad_host_range

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_amp import _amp_workload
    from tests.test_gpu_parity import _small_workload, f32, to_dev_grad, u16
    from tests import parity
else:
    dp = None

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _scratch(S):
    rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)
    assert rc == 0
    return torch.empty(max(1, nbytes // 8), dtype=torch.float64, device="cuda")


def _full_grads(wl, t):
    return [grad_host_range(wl, r, t, 0, wl.numel) for r in range(wl.n_replicas)]


def _ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


@pytest.mark.parametrize("n,S,kind", [(1, 9, 0), (2, 20_011, 0), (3, 70_001, 1), (4, 100_003, 0),
                                      (8, 50_000, 2), (13, 30_001, 0)])
def test_stored_average_matches_the_oracle(n, S, kind):
    _need_gpu()
    wl = _small_workload(n, S, kind=kind, rank=n - 1)
    gh = _full_grads(wl, 1)
    grads = [to_dev_grad(g) for g in gh]
    avg = torch.full((S,), float("nan"), device="cuda")
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    sq_ref = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = _scratch(S)
    dp.grad_average_sqnorm(grads, wl.shard_rank, avg, sq, scratch)
    dp.grad_sqnorm(grads, wl.shard_rank, sq_ref, scratch)
    dp.stream_status()
    # the norm is the one grad_sqnorm gives, bit for bit
    assert torch.equal(sq, sq_ref)
    # the average: fp64 sum in replica order, rounded to fp32, divided by N (the
    # oracle's definition); the compensated fp32 sum rounds the same way except
    # where the exact sum sits within ~2^-48 of a rounding boundary
    want = oracle.average([g[wl.shard_base:wl.shard_base + S] for g in gh])
    got = f32(avg)
    d = _ulp_diff(got, want)
    assert np.all(np.isfinite(got))
    assert d.max() <= 1
    assert (d == 0).mean() > 0.999


def _two_pass_clip(wl, steps, wd, max_norm, unscale, stored):
    S = wl.shard_elems
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    part = torch.zeros(wl.n_replicas, dtype=torch.float64, device="cuda")
    total = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = _scratch(S)
    avgs = [torch.empty(S, device="cuda") for _ in range(wl.n_replicas)]
    for t in steps:
        grads = [to_dev_grad(g) for g in _full_grads(wl, t)]
        for r in range(wl.n_replicas):
            if stored:
                dp.grad_average_sqnorm(grads, r, avgs[r], part[r:r + 1], scratch,
                                       grad_unscale=unscale)
            else:
                dp.grad_sqnorm(grads, r, part[r:r + 1], scratch, grad_unscale=unscale)
        torch.sum(part, dim=0, keepdim=True, out=total)
        opts = dp.step_options(weight_decay=wd, max_grad_norm=max_norm, grad_sqnorm=total,
                               grad_unscale=unscale)
        if stored:   # the rank's stored average as a single fp32 replica
            dp.reduce_adamw([avgs[wl.shard_rank]], 0, S, dm, dmm, dv, dout, step=t, opts=opts,
                            **HP)
        else:
            dp.reduce_adamw(grads, wl.shard_rank, S, dm, dmm, dv, dout, step=t, opts=opts, **HP)
    dp.stream_status()
    return f32(dm), f32(dmm), f32(dv), u16(dout)


@pytest.mark.parametrize("n,S,kind", [(1, 30_001, 0), (3, 20_003, 0), (4, 50_000, 0),
                                      (4, 40_000, 1), (8, 20_001, 2), (13, 9_999, 0)])
def test_two_pass_clipped_adamw_equals_the_fused_path(n, S, kind):
    _need_gpu()
    wl = _small_workload(n, S, kind=kind, rank=min(1, n - 1))
    max_norm = float(1e-4 * np.sqrt(wl.numel))   # clips: a tenth of the norm
    a = _two_pass_clip(wl, (1, 2, 3), 0.01, max_norm, 0.0, stored=True)
    b = _two_pass_clip(wl, (1, 2, 3), 0.01, max_norm, 0.0, stored=False)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_two_pass_with_unscale_equals_the_fused_path():
    _need_gpu()
    wl = _small_workload(4, 30_000, rank=2)
    a = _two_pass_clip(wl, (1, 2), 0.01, 1e-3, 2.0 ** -7, stored=True)
    b = _two_pass_clip(wl, (1, 2), 0.01, 1e-3, 2.0 ** -7, stored=False)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_two_pass_loss_scaled_run_equals_the_fused_path(max_norm):
    """Ten loss-scaled iterations with overflows at 4, 6, 7 (as in the fused
    test): the stored-average path skips, rescales and steps exactly as the
    fused path."""
    _need_gpu()
    n, S = 4, 20_000
    wl = _amp_workload(n, S)
    inject = {4: (2, 3 * S + 11, 0x7C00), 6: (0, 5, 0xFC00), 7: (3, S - 1, 0x7E00)}

    def full(k):
        bufs = [grad_host_range(wl, r, k, 0, wl.numel) for r in range(n)]
        if k in inject:
            r, i, bits = inject[k]
            bufs[r][i] = bits
        return bufs

    def run(stored):
        master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
        dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
        dout = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        state = torch.zeros(4, dtype=torch.int64, device="cuda")
        cfg = dp.loss_scale_init(state, init_scale=1024.0, window=3, hysteresis=2, min_scale=1.0)
        scratch = _scratch(S)
        part = torch.zeros(n, dtype=torch.float64, device="cuda")
        total = torch.zeros(1, dtype=torch.float64, device="cuda")
        avgs = [torch.empty(S, device="cuda") for _ in range(n)]
        trail = []
        for k in range(1, 11):
            grads = [to_dev_grad(b) for b in full(k)]
            for r in range(n):
                if stored:
                    dp.amp_average_sqnorm(grads, r, state, avgs[r], part[r:r + 1], scratch)
                else:
                    dp.amp_sqnorm(grads, r, state, part[r:r + 1], scratch)
            torch.sum(part, dim=0, keepdim=True, out=total)
            src = [avgs[wl.shard_rank]] if stored else grads
            rank = 0 if stored else wl.shard_rank
            dp.amp_step(src, rank, S, dm, dmm, dv, dout, weight_decay=0.01,
                        max_grad_norm=max_norm, global_sqnorm=total, state=state, cfg=cfg, **HP)
            st = dp.read_loss_scale(state)
            trail.append((st.scale, st.step, st.skipped, st.last_overflow))
        dp.stream_status()
        return trail, (f32(dm), f32(dmm), f32(dv), u16(dout))

    ta, a = run(True)
    tb, b = run(False)
    assert ta == tb
    assert ta[-1][2] == 3
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_stored_average_argument_checks():
    _need_gpu()
    wl = _small_workload(2, 1000)
    grads = [to_dev_grad(g) for g in _full_grads(wl, 1)]
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = _scratch(1000)
    avg = torch.empty(1001, device="cuda")
    ptrs = [g.data_ptr() for g in grads]
    nb = scratch.numel() * 8
    ok = dp.dpopt_grad_average_sqnorm(ptrs, 0, 2, 2000, 1, 0.0, avg.data_ptr(), sq.data_ptr(),
                                      scratch.data_ptr(), nb, 0)
    assert ok == dp.DPOPT_OK
    # null, misaligned, overlapping the scratch, overlapping a gradient
    for bad in (0, avg.data_ptr() + 2, scratch.data_ptr(), grads[0].data_ptr()):
        rc = dp.dpopt_grad_average_sqnorm(ptrs, 0, 2, 2000, 1, 0.0, bad, sq.data_ptr(),
                                          scratch.data_ptr(), nb, 0)
        assert rc == dp.DPOPT_ERR_INVALID_ARG, bad
    dp.stream_status()


def _contiguous_buckets(grads, base, S, bucket):
    """Bucket slices as consecutive views of the full replica buffers (a flat,
    contiguous gradient buffer), and their shard offsets."""
    rows, offs = [], []
    for off in range(0, S, bucket):
        ln = min(bucket, S - off)
        rows.append([g[base + off:base + off + ln] for g in grads])
        offs.append(off)
    return rows, offs


def _bucket_scratch(S, nb):
    rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(S, nb)
    assert rc == 0
    return torch.empty(max(1, nbytes // 8), dtype=torch.float64, device="cuda")


@pytest.mark.parametrize("n,S,bucket,kind", [(4, 100_003, 9_001, 0), (64, 40_000, 4_000, 0),
                                             (8, 50_001, 12_345, 2), (3, 30_000, 7_777, 1)])
def test_bucket_average_equals_the_full_buffer_average(n, S, bucket, kind):
    """Contiguous buckets join into one segment: the bucket norm, and the
    bucket average with its norm, are bit for bit those of the full-buffer
    entries over the same shard."""
    _need_gpu()
    wl = _small_workload(n, S, kind=kind, rank=min(2, n - 1))
    grads = [to_dev_grad(g) for g in _full_grads(wl, 1)]
    rows, offs = _contiguous_buckets(grads, wl.shard_base, S, bucket)
    sq_full, sq_b, sq_ab = (torch.zeros(1, dtype=torch.float64, device="cuda") for _ in range(3))
    avg_full = torch.full((S,), float("nan"), device="cuda")
    avg_b = torch.full((S,), float("nan"), device="cuda")
    dp.grad_average_sqnorm(grads, wl.shard_rank, avg_full, sq_full, _scratch(S))
    c0 = dp.dpopt_launch_count()
    dp.grad_sqnorm_buckets(rows, offs, sq_b, _bucket_scratch(S, len(rows)))
    assert dp.dpopt_launch_count() - c0 == 2          # one norm pass, one ordered finish
    dp.grad_average_sqnorm_buckets(rows, offs, avg_b, sq_ab, _bucket_scratch(S, len(rows)))
    dp.stream_status()
    assert torch.equal(sq_b, sq_full) and torch.equal(sq_ab, sq_full)
    assert np.array_equal(f32(avg_b).view(np.uint32), f32(avg_full).view(np.uint32))


def test_two_pass_clipped_step_over_buckets_equals_the_fused_bucket_step():
    """N = 64 in 4000-element contiguous buckets: the norm pass stores the
    average, the step reads it as one fp32 replica -- the bits of the fused
    bucket step that reads the 64 slices, step after step."""
    _need_gpu()
    n, S, bucket = 64, 40_000, 4_000
    wl = _small_workload(n, S, kind=0, rank=5)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    res = []
    for stored in (True, False):
        st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        sq = torch.zeros(1, dtype=torch.float64, device="cuda")
        avg = torch.empty(S, device="cuda")
        for t in (1, 2, 3):
            # each replica's slice of this rank's shard (what a reduce-scatter
            # hands over), one flat buffer cut into contiguous buckets
            sh = [grad_host_range(wl, r, t, wl.shard_base, S) for r in range(n)]
            grads = [to_dev_grad(g) for g in sh]
            rows, offs = _contiguous_buckets(grads, 0, S, bucket)
            scratch = _bucket_scratch(S, len(rows))
            if stored:
                dp.grad_average_sqnorm_buckets(rows, offs, avg, sq, scratch)
            else:
                dp.grad_sqnorm_buckets(rows, offs, sq, scratch)
            # this shard's norm stands for the global one here (one rank)
            opts = dp.step_options(weight_decay=0.01, max_grad_norm=1e-4 * np.sqrt(S),
                                   grad_sqnorm=sq)
            prev = tuple(f32(x) for x in st)
            if stored:
                dp.reduce_adamw([avg], 0, S, *st, out, step=t, opts=opts, **HP)
            else:
                dp.reduce_adamw_buckets(rows, offs, *st, out, step=t, opts=opts, **HP)
            dp.stream_status()
            if stored:
                c = oracle.grad_scale(oracle.grad_sqnorm(sh, 0, S, 1.0), 1e-4 * np.sqrt(S),
                                      1.0)
                parity.check_step(wl, np.arange(S), t, prev, [f32(x) for x in st] + [u16(out)],
                                  "clipped AdamW, bucket average N=64",
                                  grads_fn=lambda r, _t: sh[r], weight_decay=0.01,
                                  gscale_fn=lambda _t, _g: c)
        res.append([f32(x) for x in st] + [u16(out)])
    for x, y in zip(*res):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_bucket_average_needs_joined_buckets():
    _need_gpu()
    wl = _small_workload(4, 20_000, kind=0)
    grads = [to_dev_grad(g) for g in _full_grads(wl, 1)]
    rows, offs = _contiguous_buckets(grads, wl.shard_base, 20_000, 5_000)
    rows[2] = [x.clone() for x in rows[2]]          # bucket 2 in memory of its own
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    avg = torch.empty(20_000, device="cuda")
    c0 = dp.dpopt_launch_count()
    with pytest.raises(dp.DpoptError, match="join into one segment"):
        dp.grad_average_sqnorm_buckets(rows, offs, avg, sq, _bucket_scratch(20_000, 4))
    assert dp.dpopt_launch_count() == c0
    # the norm alone still runs over the separate pieces
    dp.grad_sqnorm_buckets(rows, offs, sq, _bucket_scratch(20_000, 4))
    dp.stream_status()
    assert float(sq.item()) > 0.0


def test_loss_scaled_run_over_buckets_equals_the_full_buffer_run():
    """The loss-scaled iterations of the two-pass test with every rank's norm
    pass over contiguous bucket slices (dpopt_amp_average_sqnorm_buckets): the
    same skips, scales and bits as the full-buffer stored-average run."""
    _need_gpu()
    n, S, bucket = 4, 20_000, 3_001
    wl = _amp_workload(n, S)
    inject = {2: (1, 3 * S + 7, 0x7C00), 5: (3, 11, 0xFC00)}

    def full(k):
        bufs = [grad_host_range(wl, r, k, 0, wl.numel) for r in range(n)]
        if k in inject:
            r, i, bits = inject[k]
            bufs[r][i] = bits
        return bufs

    def run(buckets):
        master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
        dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
        dout = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        state = torch.zeros(4, dtype=torch.int64, device="cuda")
        cfg = dp.loss_scale_init(state, init_scale=1024.0, window=2, hysteresis=2, min_scale=1.0)
        scratch = _bucket_scratch(S, -(-S // bucket))
        part = torch.zeros(n, dtype=torch.float64, device="cuda")
        total = torch.zeros(1, dtype=torch.float64, device="cuda")
        avgs = [torch.empty(S, device="cuda") for _ in range(n)]
        trail = []
        for k in range(1, 8):
            grads = [to_dev_grad(b) for b in full(k)]
            for r in range(n):
                if buckets:
                    rows, offs = _contiguous_buckets(grads, r * S, S, bucket)
                    dp.amp_average_sqnorm_buckets(rows, offs, state, avgs[r], part[r:r + 1],
                                                  scratch)
                else:
                    dp.amp_average_sqnorm(grads, r, state, avgs[r], part[r:r + 1], scratch)
            torch.sum(part, dim=0, keepdim=True, out=total)
            dp.amp_step([avgs[wl.shard_rank]], 0, S, dm, dmm, dv, dout, weight_decay=0.01,
                        max_grad_norm=1.0, global_sqnorm=total, state=state, cfg=cfg, **HP)
            st = dp.read_loss_scale(state)
            trail.append((st.scale, st.step, st.skipped, st.last_overflow))
        dp.stream_status()
        return trail, (f32(dm), f32(dmm), f32(dv), u16(dout))

    ta, a = run(True)
    tb, b = run(False)
    assert ta == tb and ta[-1][2] == 2
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_bucket_norm_does_not_depend_on_the_listing_order():
    """Buckets listed last first (the order a backward pass produces them) are
    put in shard order and joined: the norm and the stored average are bit for
    bit those of the ascending listing, and the step gives the same bits."""
    _need_gpu()
    n, S, bucket = 8, 60_001, 7_000
    wl = _small_workload(n, S, kind=0, rank=2)
    sh = [grad_host_range(wl, r, 1, wl.shard_base, S) for r in range(n)]
    grads = [to_dev_grad(g) for g in sh]
    rows, offs = _contiguous_buckets(grads, 0, S, bucket)
    res = []
    for order in (1, -1):
        r, o = rows[::order], offs[::order]
        sq = torch.zeros(1, dtype=torch.float64, device="cuda")
        sq2 = torch.zeros(1, dtype=torch.float64, device="cuda")
        avg = torch.full((S,), float("nan"), device="cuda")
        dp.grad_sqnorm_buckets(r, o, sq, _bucket_scratch(S, len(r)))
        dp.grad_average_sqnorm_buckets(r, o, avg, sq2, _bucket_scratch(S, len(r)))
        master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
        st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        c0 = dp.dpopt_launch_count()
        dp.reduce_adam_buckets(r, o, *st, out, step=1, **HP)
        assert dp.dpopt_launch_count() - c0 == 1          # joined into one segment
        dp.stream_status()
        assert torch.equal(sq, sq2)
        res.append([f32(sq), f32(avg)] + [f32(x) for x in st] + [u16(out)])
    for x, y in zip(*res):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
