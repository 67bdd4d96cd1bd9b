"""AdamW with global-norm clipping (the optimizer of the ZeRO-3 answer's
DeepSpeed example: AdamW, weight_decay 0.01, gradient_clipping 1.0) on the GPU
against the oracle: the squared-norm pre-pass, the clipped AdamW step, and
the plain-Adam special cases."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.parity import grad_host_range, oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import _host_full_buffers, _small_workload, f32, to_dev_grad, u16
else:
    dp = None

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _scratch(elems, nb=1):
    rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(elems, nb)
    assert rc == 0
    return torch.empty(max(1, nbytes // 8), dtype=torch.float64, device="cuda")


@pytest.mark.parametrize("n,S,kind", [(1, 5, 0), (4, 65536, 0), (3, 200_003, 0), (8, 131_073, 1),
                                      (64, 70_001, 0), (13, 1_000_000, 0)])
def test_sqnorm_matches_the_oracle(n, S, kind):
    _need_gpu()
    wl = _small_workload(n, S, kind=kind, rank=n - 1)
    gh = _host_full_buffers(wl, 1)
    grads = [to_dev_grad(g) for g in gh]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = _scratch(S)
    for unscale in (0.0, 0.125):
        dp.grad_sqnorm(grads, wl.shard_rank, out, scratch, grad_unscale=unscale)
        dp.stream_status()
        want = oracle.grad_sqnorm(gh, wl.shard_base, S, unscale or 1.0)
        # both sums round: the oracle's sequential fp64 sum of S terms is within
        # S * 2^-53 (relative, all terms >= 0) of the exact one, the GPU's within less
        assert float(out.item()) == pytest.approx(want, rel=4 * S * 2.0 ** -53, abs=1e-300)
    # bitwise reproducible run to run
    a = out.clone()
    dp.grad_sqnorm(grads, wl.shard_rank, out, scratch, grad_unscale=0.125)
    dp.stream_status()
    assert torch.equal(a, out)


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_sqnorm_every_unrolled_replica_count(n, kind):
    """The norm pass has a kernel per N = 1..8 and a runtime-count one above."""
    _need_gpu()
    S = 140_003
    wl = _small_workload(n, S, kind=kind, rank=0)
    gh = _host_full_buffers(wl, 1)
    grads = [to_dev_grad(g) for g in gh]
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_sqnorm(grads, wl.shard_rank, out, _scratch(S))
    dp.stream_status()
    want = oracle.grad_sqnorm(gh, wl.shard_base, S, 1.0)
    assert float(out.item()) == pytest.approx(want, rel=4 * S * 2.0 ** -53, abs=1e-300)


def test_sqnorm_over_bucket_slices_matches_full_buffer():
    _need_gpu()
    wl = _small_workload(4, 300_000, rank=1)
    gh = _host_full_buffers(wl, 1)
    grads = [to_dev_grad(g) for g in gh]
    S, base = wl.shard_elems, wl.shard_base
    full = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_sqnorm(grads, 1, full, _scratch(S))
    rows, offs = [], []
    for off in range(0, S, 70_000):
        ln = min(70_000, S - off)
        rows.append([g[base + off:base + off + ln] for g in grads])
        offs.append(off)
    part = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_sqnorm_buckets(rows, offs, part, _scratch(S, len(rows)))
    dp.stream_status()
    # the slices continue one another: joined into the full buffer's one segment,
    # they take its chunk partition and give its bits
    assert torch.equal(part, full)


def _clipped_run(wl, steps, wd, max_norm, unscale=0.0):
    """Every rank's sqnorm on the GPU, summed (the one-scalar all-reduce a
    multi-rank run does), then the clipped AdamW step of this rank's shard."""
    S = wl.shard_elems
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    total = torch.zeros(1, dtype=torch.float64, device="cuda")
    part = torch.zeros(wl.n_replicas, dtype=torch.float64, device="cuda")
    scratch = _scratch(S)
    for t in steps:
        prev = (f32(dm), f32(dmm), f32(dv))
        host = _full_grads(wl, t)
        grads = [to_dev_grad(g) for g in host]
        for r in range(wl.n_replicas):
            dp.grad_sqnorm(grads, r, part[r:r + 1], scratch, grad_unscale=unscale)
        torch.sum(part, dim=0, keepdim=True, out=total)
        opts = dp.step_options(weight_decay=wd, max_grad_norm=max_norm, grad_sqnorm=total,
                               grad_unscale=unscale)
        dp.reduce_adamw(grads, wl.shard_rank, S, dm, dmm, dv, dout, step=t, opts=opts, **HP)
        dp.stream_status()
        # step t on its own, from the GPU's previous states
        un = unscale if unscale else 1.0
        c = oracle.grad_scale(oracle.grad_sqnorm(host, 0, wl.numel, un), max_norm, un)
        parity.check_step(wl, np.arange(S), t, prev, (f32(dm), f32(dmm), f32(dv), u16(dout)),
                          f"adamw+clip N={wl.n_replicas} S={S}", weight_decay=wd,
                          gscale_fn=lambda _t, _g: c)
    dp.stream_status()
    return f32(dm), f32(dmm), f32(dv), u16(dout)


def _full_grads(wl, t):
    """Complete replica buffers (every rank's shard filled): clipping needs the
    global norm."""
    return [grad_host_range(wl, r, t, 0, wl.numel) for r in range(wl.n_replicas)]


def _oracle_clipped(wl, steps, wd, max_norm, unscale=1.0):
    def gscale(t, _grads):
        full = _full_grads(wl, t)
        sq = oracle.grad_sqnorm(full, 0, wl.numel, unscale)
        return oracle.grad_scale(sq, max_norm, unscale)
    return oracle_trajectory(wl, np.arange(wl.shard_elems), steps[0], steps[-1],
                             weight_decay=wd, gscale_fn=gscale)


@pytest.mark.parametrize("n,S", [(1, 30_001), (2, 30_001), (3, 20_003), (4, 50_000),
                                 (5, 12_007), (6, 10_001), (7, 9_001), (8, 20_001),
                                 (16, 9_999), (24, 5_003), (64, 2_011)])
def test_clipped_adamw_matches_the_oracle(n, S):
    _need_gpu()
    wl = _small_workload(n, S, rank=min(1, n - 1))
    # the averaged gradient's global norm is ~1e-3*sqrt(numel/n): clip to a tenth of it
    max_norm = float(1e-4 * np.sqrt(wl.numel))
    refs = _oracle_clipped(wl, (1, 2, 3), 0.01, max_norm)
    got = _clipped_run(wl, (1, 2, 3), 0.01, max_norm)
    st = parity.check(refs[-1], *got, where=f"adamw+clip N={n}")
    assert st.bitwise_master > 0.999


def test_power_of_two_unscale_with_clipping_matches_the_oracle():
    _need_gpu()
    wl = _small_workload(4, 30_000, rank=2)
    refs = _oracle_clipped(wl, (1, 2), 0.01, 1e-3, unscale=2.0 ** -7)
    got = _clipped_run(wl, (1, 2), 0.01, 1e-3, unscale=2.0 ** -7)
    parity.check(refs[-1], *got, where="unscale+clip")


def test_inactive_options_reproduce_plain_adam():
    """weight_decay 0 and a clip threshold far above the norm: the extended
    kernel gives the values plain Adam gives."""
    _need_gpu()
    wl = _small_workload(4, 40_000, rank=0)
    a = _clipped_run(wl, (1, 2), 0.0, 1e30)
    from tests.test_gpu_parity import _run_small_full
    # _run_small_full uses NaN outside the shard; same shard values
    b = _run_small_full(wl, steps=(1, 2))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_options_are_validated():
    _need_gpu()
    wl = _small_workload(2, 1000)
    grads = [to_dev_grad(g) for g in _host_full_buffers(wl, 1)]
    st = [torch.zeros(1000, device="cuda") for _ in range(3)]
    o = torch.zeros(1000, dtype=torch.bfloat16, device="cuda")
    for bad in (dp.step_options(weight_decay=-1.0), dp.step_options(max_grad_norm=1.0),
                dp.step_options(grad_unscale=float("inf"))):
        with pytest.raises(dp.DpoptError):
            dp.reduce_adamw(grads, 1, 1000, *st, o, step=1, opts=bad, **HP)
