"""The step entries inside captured CUDA graphs.

Every entry only enqueues work on its stream and never synchronises, so it can
be captured.  The loss-scaled entries keep the step count and the scale on the
device, so one graph of a whole iteration (norm passes, the scalar sum, the
step, the scale update) replays iteration after iteration: K replays must give
the bits of K direct calls, overflow skips included.  With no squared norm the
same step is a run without loss scaling whose step count lives on the device,
checked step by step against the oracle.  Entries that take the step from the
caller replay that step; the table entry refuses to be captured when it would
copy its launch table from reused host memory.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.parity import grad_host_range

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_amp import _amp_workload
    from tests.test_gpu_parity import HP, _small_workload, f32, to_dev_grad, u16
    from tests.test_gpu_table import _slices
else:
    dp = None


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class _Iteration:
    """Static buffers of one rank's loss-scaled iteration: N replica gradient
    buffers (refilled before every iteration), the shard's states, the
    loss-scale state, the per-rank norms and their sum."""

    def __init__(self, wl, master, m, v, cfg_args, max_norm):
        n, S = wl.n_replicas, wl.shard_elems
        dt = torch.float16 if wl.grad_kind == 2 else torch.bfloat16
        self.wl, self.max_norm = wl, max_norm
        self.grads = [torch.zeros(wl.numel, dtype=dt, device="cuda") for _ in range(n)]
        self.st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        self.out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
        self.state = torch.zeros(4, dtype=torch.int64, device="cuda")
        self.cfg = dp.loss_scale_init(self.state, **cfg_args)
        rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)
        assert rc == dp.DPOPT_OK
        self.scratch = torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")
        self.part = torch.zeros(n, dtype=torch.float64, device="cuda")
        self.total = torch.zeros(1, dtype=torch.float64, device="cuda")

    def fill(self, host):
        for g, h in zip(self.grads, host):
            g.copy_(to_dev_grad(h))

    def run(self):
        """The iteration on the current stream: every rank's norm (their sum is
        the one-scalar all-reduce), then the step and the scale update."""
        wl = self.wl
        for r in range(wl.n_replicas):
            dp.amp_sqnorm(self.grads, r, self.state, self.part[r:r + 1], self.scratch)
        torch.sum(self.part, dim=0, keepdim=True, out=self.total)
        dp.amp_step(self.grads, wl.shard_rank, wl.shard_elems, *self.st, self.out,
                    weight_decay=0.01, max_grad_norm=self.max_norm, global_sqnorm=self.total,
                    state=self.state, cfg=self.cfg, **HP)

    def snapshot(self):
        return [f32(x) for x in self.st] + [u16(self.out)]


@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_loss_scaled_iteration_replays_from_one_graph(max_norm):
    _need_gpu()
    n, S = 4, 30_011
    wl = _amp_workload(n, S)
    inject = {3: (1, 2 * S + 5, 0x7C00), 5: (0, 17, 0xFC00), 6: (2, S + 1, 0x7E00)}

    def full(k):
        bufs = [grad_host_range(wl, r, k, 0, wl.numel) for r in range(n)]
        if k in inject:
            r, i, bits = inject[k]
            bufs[r][i] = bits
        return bufs

    cfg_args = dict(init_scale=1024.0, window=2, hysteresis=2, min_scale=1.0)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    direct = _Iteration(wl, master, m, v, cfg_args, max_norm)
    replay = _Iteration(wl, master, m, v, cfg_args, max_norm)
    warm = _Iteration(wl, master, m, v, cfg_args, max_norm)
    warm.fill(full(1))
    warm.run()             # loads every kernel of the iteration before the capture
    dp.stream_status()
    c0 = dp.dpopt_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        replay.run()
    per_iteration = dp.dpopt_launch_count() - c0
    assert per_iteration == 2 * n + 2     # n norm passes + finishes, the step, the update
    K = 8
    refs = parity.oracle_amp_trajectory(
        wl, K, full, oracle.LossScaler(1024.0, 2, 2, 1.0), weight_decay=0.01,
        max_grad_norm=max_norm)
    for k in range(1, K + 1):
        host = full(k)
        direct.fill(host)
        direct.run()
        replay.fill(host)
        c0 = dp.dpopt_launch_count()
        graph.replay()
        assert dp.dpopt_launch_count() == c0      # a replay goes through no entry point
        dp.stream_status()
        a, b = direct.snapshot(), replay.snapshot()
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), k
        sa, sb = dp.read_loss_scale(direct.state), dp.read_loss_scale(replay.state)
        assert (sa.scale, sa.step, sa.skipped, sa.last_overflow) == \
               (sb.scale, sb.step, sb.skipped, sb.last_overflow), k
        _, overflow, scale, steps = refs[k - 1]
        assert (bool(sb.last_overflow), sb.scale, sb.step) == (overflow, scale, steps), k
    parity.check(refs[-1][0], *replay.snapshot(), where=f"graph amp max_norm={max_norm}")
    assert sb.skipped == 3


def test_device_step_count_without_loss_scaling_replays():
    """amp_step with no squared norm: no overflow test, the scale left at 1, the
    step count advanced on the device.  One captured step replayed four times
    is four AdamW steps, each checked on its own against the oracle."""
    _need_gpu()
    n, S = 8, 50_001
    wl = _small_workload(n, S, kind=0, rank=3)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    it = _Iteration(wl, master, m, v, dict(init_scale=1.0, window=1, hysteresis=1,
                                           min_scale=1.0), 0.0)
    warm = _Iteration(wl, master, m, v, dict(init_scale=1.0, window=1, hysteresis=1,
                                             min_scale=1.0), 0.0)

    def step(x):
        dp.amp_step(x.grads, wl.shard_rank, S, *x.st, x.out, weight_decay=0.01,
                    max_grad_norm=0.0, global_sqnorm=None, state=x.state, cfg=x.cfg, **HP)

    step(warm)
    dp.stream_status()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(it)
    base = wl.shard_base
    for t in range(1, 5):
        host = [grad_host_range(wl, r, t, 0, wl.numel) for r in range(n)]
        prev = tuple(f32(x) for x in it.st)
        it.fill(host)
        graph.replay()
        dp.stream_status()
        st = dp.read_loss_scale(it.state)
        assert (st.step, st.scale, st.skipped, st.last_overflow) == (t, 1.0, 0, 0)
        parity.check_step(wl, np.arange(S), t, prev, it.snapshot(), "graph, device step count",
                          grads_fn=lambda r, _t: host[r][base:base + S], weight_decay=0.01)


def test_learning_rate_schedule_from_device_memory_replays():
    """The step reads its learning rate from device memory: one captured step,
    the rate rewritten before every replay (a warm-up then decay schedule),
    each replayed step against the oracle at that step's rate, and bit for bit
    the direct calls that pass the same rates from the host."""
    _need_gpu()
    n, S = 4, 30_007
    wl = _small_workload(n, S, kind=0, rank=1)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    cfg = dict(init_scale=1.0, window=1, hysteresis=1, min_scale=1.0)
    rates = [float(np.float32(x)) for x in (2e-4, 6e-4, 1e-3, 7e-4, 3e-4)]
    lr_dev = torch.zeros(1, device="cuda")
    hp = dict(beta1=HP["beta1"], beta2=HP["beta2"], eps=HP["eps"])

    def step(x, **kw):
        dp.amp_step(x.grads, wl.shard_rank, S, *x.st, x.out, weight_decay=0.05,
                    max_grad_norm=0.0, global_sqnorm=None, state=x.state, cfg=x.cfg, **hp, **kw)

    warm = _Iteration(wl, master, m, v, cfg, 0.0)
    step(warm, lr=0.0, lr_dev=lr_dev)
    dp.stream_status()
    it = _Iteration(wl, master, m, v, cfg, 0.0)
    direct = _Iteration(wl, master, m, v, cfg, 0.0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(it, lr=float("nan"), lr_dev=lr_dev)    # the host rate is not used
    base = wl.shard_base
    for t, lr in enumerate(rates, start=1):
        host = [grad_host_range(wl, r, t, 0, wl.numel) for r in range(n)]
        prev = tuple(f32(x) for x in it.st)
        it.fill(host)
        direct.fill(host)
        lr_dev.fill_(lr)
        graph.replay()
        step(direct, lr=lr)
        dp.stream_status()
        got = it.snapshot()
        for x, y in zip(got, direct.snapshot()):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), t
        parity.check_step(wl, np.arange(S), t, prev, got, "graph, device learning rate",
                          grads_fn=lambda r, _t: host[r][base:base + S],
                          hp=dict(lr=lr, **hp), weight_decay=0.05)


def test_clipping_without_a_norm_is_refused():
    _need_gpu()
    wl = _small_workload(2, 1_000, kind=0)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(1_000))
    it = _Iteration(wl, master, m, v, dict(init_scale=1.0, window=1, hysteresis=1,
                                           min_scale=1.0), 1.0)
    c0 = dp.dpopt_launch_count()
    with pytest.raises(dp.DpoptError):
        dp.amp_step(it.grads, wl.shard_rank, 1_000, *it.st, it.out, weight_decay=0.0,
                    max_grad_norm=1.0, global_sqnorm=None, state=it.state, cfg=it.cfg, **HP)
    assert dp.dpopt_launch_count() == c0


def test_caller_step_entries_replay_their_step():
    """The plain entry captured at step t: a replay is that step again, with
    the bits of the direct call."""
    _need_gpu()
    n, S = 4, 40_007
    wl = _small_workload(n, S, kind=0)
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    host = [grad_host_range(wl, r, 3, 0, wl.numel) for r in range(n)]
    grads = [to_dev_grad(h) for h in host]
    res = []
    for mode in ("direct", "graph"):
        st = [torch.from_numpy(x.copy()).cuda() for x in (master, m, v)]
        out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")

        def call():
            dp.reduce_adam(grads, wl.shard_rank, S, *st, out, step=3, **HP)

        if mode == "direct":
            call()
        else:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                call()
            assert not st[1].ne(torch.from_numpy(m).cuda()).any()   # captured, not run
            graph.replay()
        dp.stream_status()
        res.append([f32(x) for x in st] + [u16(out)])
    for x, y in zip(*res):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_table_entry_refuses_capture_when_it_writes_the_table():
    _need_gpu()
    wl = _small_workload(64, 40_003, kind=0)
    rows, offs = _slices(wl, 1, 997)       # 41 buckets x 64 separate slices: a table
    S = wl.shard_elems
    st = [torch.zeros(S, device="cuda") for _ in range(3)]
    out = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
    table = torch.empty(dp.bucket_table_bytes(64, len(rows)), dtype=torch.uint8, device="cuda")
    other = torch.zeros(1, device="cuda")
    graph = torch.cuda.CUDAGraph()
    c0 = dp.dpopt_launch_count()
    with torch.cuda.graph(graph):
        other.add_(1.0)                    # the rest of the capture goes on
        with pytest.raises(dp.DpoptError, match="captured graph"):
            dp.reduce_adam_buckets_table(rows, offs, *st, out, table, step=1, **HP)
    assert dp.dpopt_launch_count() == c0
    graph.replay()
    torch.cuda.synchronize()
    assert other.item() == 1.0 and not st[0].any()
    # outside a capture the same call runs
    dp.reduce_adam_buckets_table(rows, offs, *st, out, table, step=1, **HP)
    dp.stream_status()
    assert st[2].any()
