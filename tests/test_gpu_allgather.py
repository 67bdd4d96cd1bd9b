"""ZeRO-3 parameter all-gather on one GPU: after every rank's shard step and
all-gather, every replica's bf16 parameters equal the data-parallel update."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from tests import parity

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import _host_full_buffers, _small_workload, f32, to_dev_grad, u16
    from tests.parity import oracle_trajectory
else:
    dp = None

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("n,S", [(4, 50_000), (3, 7), (8, 10_001), (64, 2_048)])
def test_every_replica_ends_with_the_data_parallel_parameters(n, S):
    _need_gpu()
    numel = n * S
    wl = _small_workload(n, S, rank=0)
    rng = np.random.default_rng(n * S)
    gh = [oracle.f32_to_bf16((rng.standard_normal(numel) * 1e-3).astype(np.float32))
          for _ in range(n)]
    th0 = (rng.standard_normal(numel) * 0.02).astype(np.float32)
    grads = [to_dev_grad(g) for g in gh]
    replicas = [torch.full((numel,), float("nan"), dtype=torch.bfloat16, device="cuda")
                for _ in range(n)]
    for r in range(n):   # every rank: its shard's step, then the all-gather of its shard
        st = [torch.from_numpy(th0[r * S:(r + 1) * S].copy()).cuda(),
              torch.zeros(S, device="cuda"), torch.zeros(S, device="cuda")]
        out = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        dp.reduce_adam(grads, r, S, *st, out, step=1, **HP)
        dp.allgather_bf16(out, r, replicas)
    dp.stream_status()
    # the oracle's data-parallel update of the whole vector
    m = np.zeros(numel, np.float32)
    v = np.zeros(numel, np.float32)
    th = th0.copy()
    want = oracle.reduce_adam_range(gh, 0, numel, th, m, v, step=1, **HP)
    for rep in replicas:
        got = u16(rep)
        d = np.abs(parity.bf16_ordered(got) - parity.bf16_ordered(want))
        assert d.max() <= 1 and np.mean(got == want) > 0.999


def test_unaligned_and_self_aliased_destinations():
    _need_gpu()
    n, S = 3, 1001
    base = [torch.zeros(n * S + 8, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    reps = [b[1:1 + n * S] for b in base]          # 2-byte aligned only: scalar path
    shard = torch.arange(S, dtype=torch.float32, device="cuda").to(torch.bfloat16)
    dp.allgather_bf16(shard, 2, reps)
    # the shard already in replica 1's slot is skipped, the others are written
    reps[1][2 * S:3 * S] = shard
    dp.allgather_bf16(reps[1][2 * S:3 * S], 2, reps)
    dp.stream_status()
    want = u16(shard)
    for rep in reps:
        np.testing.assert_array_equal(u16(rep[2 * S:3 * S]), want)
        assert not rep[:2 * S].float().any()
    for b in base:
        assert b[0].item() == 0 and not b[1 + n * S:].float().any()


def test_allgather_rejects_bad_arguments():
    _need_gpu()
    x = torch.zeros(100, dtype=torch.bfloat16, device="cuda")
    reps = [torch.zeros(200, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    P = x.data_ptr()
    R = [r.data_ptr() for r in reps]
    assert dp.dpopt_allgather_bf16(P, 100, 2, R, 2, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_allgather_bf16(P, 100, 0, [R[0], R[0] + 20], 2, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_allgather_bf16(R[0] + 10, 100, 0, R, 2, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_allgather_bf16(P + 1, 100, 0, R, 2, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_allgather_bf16(P, 100, 0, R, 65, 0) == dp.DPOPT_ERR_UNSUPPORTED


def _states(wl):
    """The rank's seeded master, m, v on the device."""
    th, m, v = parity.states_host(wl, np.arange(wl.shard_elems) + wl.shard_base)
    return [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (th, m, v)]


@pytest.mark.parametrize("n,S,kind,rank", [
    (1, 4_099, 0, 0), (2, 50_001, 0, 1), (3, 30_000, 0, 2), (4, 65_537, 0, 1),
    (5, 12_345, 0, 3), (8, 20_003, 0, 7), (13, 4_100, 0, 6), (64, 2_056, 0, 17),
    (4, 40_000, 1, 2), (2, 9_999, 1, 0), (4, 30_011, 2, 3),
])
def test_fused_step_allgather_equals_step_then_allgather(n, S, kind, rank):
    """Two steps of the fused entry against the step followed by the separate
    all-gather: the same master/m/v and the same bytes in every replica buffer
    (canary-filled outside the shard), and the oracle's values on a sample."""
    _need_gpu()
    wl = _small_workload(n, S, kind=kind, rank=rank, seed=23)
    numel = n * S
    res = []
    idx = np.unique(np.concatenate([np.arange(0, S, 97), np.arange(max(0, S - 9), S)]))
    for fused in (True, False):
        st = _states(wl)
        reps = [torch.full((numel,), 0x7FA1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
                for _ in range(n)]   # a NaN bit pattern no step writes
        for t in (1, 2):
            prev = [f32(x)[idx] for x in st]
            grads = [to_dev_grad(g) for g in _host_full_buffers(wl, t)]
            if fused:
                dp.reduce_adam_allgather(grads, rank, S, *st, reps, step=t, **HP)
                dp.stream_status()
                got = [f32(x)[idx] for x in st] + [u16(reps[(rank + 1) % n])[rank * S + idx]]
                parity.check_step(wl, idx, t, prev, got, f"fused gather N={n} S={S}")
            else:
                own = reps[rank][rank * S:(rank + 1) * S]
                dp.reduce_adam(grads, rank, S, *st, own, step=t, **HP)
                dp.allgather_bf16(own, rank, reps)
        dp.stream_status()
        res.append([f32(x) for x in st] + [u16(r) for r in reps])
    for a, b in zip(*res):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    ref = oracle_trajectory(wl, idx, 1, 2)[-1]
    th, m, v = (x[idx] for x in res[0][:3])
    for r in range(n):
        parity.check(ref, th, m, v, res[0][3 + r][rank * S + idx], where=f"fused gather rep {r}")
        outside = np.concatenate([res[0][3 + r][:rank * S], res[0][3 + r][(rank + 1) * S:]])
        assert (outside == 0x7FA1).all()


def test_fused_step_allgather_unaligned_replicas():
    """Replica buffers 2 bytes past a 16-byte boundary: the one-element path,
    same bits as the separate step and all-gather."""
    _need_gpu()
    n, S, rank = 3, 10_007, 1
    wl = _small_workload(n, S, rank=rank, seed=29)
    grads = [to_dev_grad(g) for g in _host_full_buffers(wl, 1)]
    res = []
    for fused in (True, False):
        st = _states(wl)
        base = [torch.zeros(n * S + 8, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        reps = [b[1:1 + n * S] for b in base]
        if fused:
            dp.reduce_adam_allgather(grads, rank, 1000, *st, reps, step=1, **HP)
        else:
            own = reps[rank][rank * S:(rank + 1) * S]
            dp.reduce_adam(grads, rank, 1000, *st, own, step=1, **HP)
            dp.allgather_bf16(own, rank, reps)
        dp.stream_status()
        res.append([f32(x) for x in st] + [u16(b) for b in base])
    for a, b in zip(*res):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("n,S", [(4, 13_000_000), (8, 9_200_001), (12, 7_200_000)])
def test_large_shard_entry_writes_the_bits_of_the_two_calls(n, S):
    """Shards whose working set is far above L2 (0.9-1.2 GB), where whole 4 KB
    tiles go to the replicas by bulk copies: the entry writes the bits of the
    step into the own replica followed by the broadcast (the two public
    calls)."""
    _need_gpu()
    rank = n - 1
    gen = torch.Generator(device="cuda")
    gen.manual_seed(n)
    grads = [torch.randn(n * S, generator=gen, device="cuda").mul_(1e-3).bfloat16()
             for _ in range(n)]
    init = [torch.randn(S, generator=gen, device="cuda").mul_(0.02),
            torch.randn(S, generator=gen, device="cuda").mul_(1e-4),
            torch.randn(S, generator=gen, device="cuda").mul_(1e-6).abs()]
    res = []
    for fused in (True, False):
        st = [x.clone() for x in init]
        reps = [torch.full((n * S,), 0x7FA1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
                for _ in range(n)]
        if fused:
            dp.reduce_adam_allgather(grads, rank, S, *st, reps, step=3, **HP)
        else:
            own = reps[rank][rank * S:(rank + 1) * S]
            dp.reduce_adam(grads, rank, S, *st, own, step=3, **HP)
            dp.allgather_bf16(own, rank, reps)
        dp.stream_status()
        res.append([x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16)
                    for x in st + reps])
        del reps
    for a, b in zip(*res):
        assert torch.equal(a, b)


@pytest.mark.parametrize("n,S", [(2, 50_001), (5, 100_003), (13, 20_007)])
def test_gather_policies_write_the_same_bits(n, S):
    """The fused kernel and the two-pass form, forced by the gather policy,
    leave the same states and replica buffers as the automatic choice."""
    _need_gpu()
    rank = n // 2
    gen = torch.Generator(device="cuda")
    gen.manual_seed(100 + n)
    grads = [torch.randn(n * S, generator=gen, device="cuda").mul_(1e-3).bfloat16()
             for _ in range(n)]
    init = [torch.randn(S, generator=gen, device="cuda").mul_(0.02),
            torch.randn(S, generator=gen, device="cuda").mul_(1e-4),
            torch.randn(S, generator=gen, device="cuda").mul_(1e-6).abs()]
    res = []
    for pol in (dp.DPOPT_GATHER_AUTO, dp.DPOPT_GATHER_FUSED, dp.DPOPT_GATHER_SEPARATE):
        st = [x.clone() for x in init]
        reps = [torch.full((n * S,), 0x7FA1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
                for _ in range(n)]
        with dp.gather_policy(pol):
            for t in (1, 2):
                dp.reduce_adam_allgather(grads, rank, S, *st, reps, step=t, **HP)
        dp.stream_status()
        res.append([x.view(torch.int32) for x in st] + [r.view(torch.int16) for r in reps])
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)
    assert dp.dpopt_get_gather_policy() == dp.DPOPT_GATHER_AUTO
