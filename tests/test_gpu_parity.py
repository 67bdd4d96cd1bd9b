"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Small cases compare every element; the full-size workloads compare sampled
elements (bucket edges, the ragged tail, and seeded random picks) that the
oracle computes one by one from the same seeded inputs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from synth.device import DeviceWorkload, workload_bytes
from tests import parity
from tests.parity import grad_host_range, oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
else:  # collected on a CPU-only machine: every test here is skipped by the marker run
    dp = None


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def to_dev_grad(a: np.ndarray, dev="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        dt = torch.float16 if isinstance(a, oracle.F16Bits) else torch.bfloat16
        return torch.from_numpy(np.asarray(a).view(np.int16).copy()).to(dev).view(dt)
    return torch.from_numpy(a.copy()).to(dev)


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _small_workload(n, S, kind=0, rank=None, dist=None, seed=11):
    return synth.Workload(name=f"small_N{n}_S{S}", n_replicas=n, numel=n * S,
                          shard_rank=(n - 1) if rank is None else rank, bucket_elems=max(1, S),
                          seed=seed, grad_dist=lambda r: dist or synth.Dist(r * 1e-5, 1e-3),
                          master_dist=synth.Dist(0.0, 0.02), m_dist=synth.Dist(0.0, 1e-4),
                          v_dist=synth.Dist(0.0, 1e-6, absval=True), steps=2, grad_kind=kind)


def _host_full_buffers(wl, t):
    """N full replica buffers: the rank's shard holds step t's seeded gradients,
    everything else NaN (a read outside the shard would poison the result)."""
    out = []
    for r in range(wl.n_replicas):
        if wl.grad_kind == 0:
            buf = np.full(wl.numel, 0x7FC0, dtype=np.uint16)
        elif wl.grad_kind == 2:
            buf = oracle.as_f16_bits(np.full(wl.numel, 0x7E00, dtype=np.uint16))
        else:
            buf = np.full(wl.numel, np.nan, dtype=np.float32)
        buf[wl.shard_base:wl.shard_base + wl.shard_elems] = grad_host_range(
            wl, r, t, wl.shard_base, wl.shard_elems)
        out.append(buf)
    return out


def _run_small_full(wl, steps=(1, 2), entry="full", bucket=None, hp=HP, per_step=True):
    """Host-generated inputs, uploaded; returns final device states as numpy.
    per_step: every step is also checked on its own against one oracle step
    from the GPU's previous states (the stated per-value bound)."""
    S = wl.shard_elems
    gidx = wl.shard_base + np.arange(S, dtype=np.int64)
    master, m, v = parity.states_host(wl, gidx)
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    for t in steps:
        prev = (f32(dm), f32(dmm), f32(dv)) if per_step else None
        grads = [to_dev_grad(g) for g in _host_full_buffers(wl, t)]
        if entry == "full":
            dp.reduce_adam(grads, wl.shard_rank, bucket or wl.bucket_elems, dm, dmm, dv, dout,
                           step=t, **hp)
        elif entry == "bucket":
            be = bucket or S
            for off in range(0, S, be):
                ln = min(be, S - off)
                sl = [g[wl.shard_base + off:wl.shard_base + off + ln] for g in grads]
                dp.reduce_adam_bucket(sl, off, dm, dmm, dv, dout, step=t, **hp)
        else:
            be = bucket or S
            rows, offs = [], []
            for off in range(0, S, be):
                ln = min(be, S - off)
                rows.append([g[wl.shard_base + off:wl.shard_base + off + ln] for g in grads])
                offs.append(off)
            dp.reduce_adam_buckets(rows, offs, dm, dmm, dv, dout, step=t, **hp)
        if per_step:
            dp.stream_status()
            parity.check_step(wl, np.arange(S), t, prev, (f32(dm), f32(dmm), f32(dv), u16(dout)),
                              _config_name(wl), hp=hp)
    dp.stream_status()
    return f32(dm), f32(dmm), f32(dv), u16(dout)


def _config_name(wl):
    kind = ("bf16", "fp32", "fp16")[wl.grad_kind]
    return f"N={wl.n_replicas} S={wl.shard_elems} {kind}"


# ---------------------------------------------------------------------------
# generator twin
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [0, 1])
def test_device_generator_matches_host_generator(kind):
    _need_gpu()
    d = synth.Dist(1e-5, 1e-3, outlier_p=0.01, outlier_scale=100.0)
    n, start = 1_000_003, 123_456_789
    buf = torch.empty(n, dtype=torch.bfloat16 if kind == 0 else torch.float32, device="cuda")
    synth.device_fill(buf.data_ptr(), kind, start, n, 7, 99, d)
    torch.cuda.synchronize()
    got = u16(buf) if kind == 0 else f32(buf)
    want = synth.host_fill(kind, start, n, 7, 99, d)
    np.testing.assert_array_equal(got.view(np.uint16 if kind == 0 else np.uint32),
                                  want.view(np.uint16 if kind == 0 else np.uint32))


# ---------------------------------------------------------------------------
# small cases: every element
# ---------------------------------------------------------------------------

def test_tiny_every_element_three_steps():
    _need_gpu()
    wl = synth.WORKLOADS["tiny"]
    S = wl.shard_elems
    refs = oracle_trajectory(wl, np.arange(S), 1, wl.steps)
    dev = DeviceWorkload(wl)
    dev.fill_states()
    for t in range(1, wl.steps + 1):
        prev = (f32(dev.master), f32(dev.m), f32(dev.v))
        dev.fill_grads(t)
        dp.reduce_adam(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m, dev.v,
                       dev.out, lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=t)
        dp.stream_status()
        got = (f32(dev.master), f32(dev.m), f32(dev.v), u16(dev.out))
        parity.check(refs[t - 1], *got, where=f"tiny t={t}")
        parity.check_step(wl, np.arange(S), t, prev, got, "tiny")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 13, 64])
@pytest.mark.parametrize("S", [1, 7, 8, 15, 4097, 100_003])
def test_ragged_sizes_every_element(n, S):
    _need_gpu()
    wl = _small_workload(n, S)
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    got = _run_small_full(wl, steps=(1, 2))
    parity.check(refs[-1], *got, where=f"N={n} S={S}")


@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9])
def test_every_unrolled_replica_count(n, kind):
    """N = 1..8 each run their own kernel (replica loop unrolled), N = 9 the
    runtime-count body: every element of a ragged shard agrees with the oracle
    for bf16, fp32 and fp16 gradients, and the batched-bucket entry (the other
    segment table) gives the same bits."""
    _need_gpu()
    S = 20_011
    wl = _small_workload(n, S, kind=kind)
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    got = _run_small_full(wl, steps=(1, 2))
    parity.check(refs[-1], *got, where=f"N={n} kind={kind}")
    got_b = _run_small_full(wl, steps=(1, 2), entry="buckets", bucket=4_099)
    for x, y in zip(got, got_b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("kind", [0, 2])
@pytest.mark.parametrize("n", [17, 18, 20, 21, 24, 40, 56, 57, 63, 64])
def test_many_replicas_both_walks_every_element(n, kind):
    """16-bit gradients with many replicas: N = 17..20 take unrolled kernels
    (three batches of loads), N = 21..63 the walk that stages the replica loads
    in shared memory, N = 64 the register-pipelined walk; every element
    agrees with the oracle step by step, and the batched-bucket entry gives
    the same bits."""
    _need_gpu()
    S = 9_001
    wl = _small_workload(n, S, kind=kind)
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    got = _run_small_full(wl, steps=(1, 2))
    parity.check(refs[-1], *got, where=f"N={n} kind={kind}")
    got_b = _run_small_full(wl, steps=(1, 2), entry="buckets", bucket=2_003)
    for x, y in zip(got, got_b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 13])
@pytest.mark.parametrize("S", [9, 40_000])
def test_fp32_gradients_every_element(n, S):
    _need_gpu()
    wl = _small_workload(n, S, kind=1)
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    got = _run_small_full(wl, steps=(1, 2))
    parity.check(refs[-1], *got, where=f"fp32 N={n} S={S}")


@pytest.mark.parametrize("hp", [
    dict(lr=1e-2, beta1=0.8, beta2=0.95, eps=1e-3),
    dict(lr=3e-4, beta1=0.0, beta2=0.0, eps=0.0),
    dict(lr=1e-3, beta1=0.3, beta2=0.6, eps=1e-12),
    dict(lr=-1e-3, beta1=0.99, beta2=0.9999, eps=1e-6),
])
def test_other_hyperparameters_every_element(hp):
    _need_gpu()
    wl = _small_workload(4, 20_011)
    refs = oracle_trajectory(wl, np.arange(wl.shard_elems), 1, 3, hp=hp)
    got = _run_small_full(wl, steps=(1, 2, 3), hp=hp)
    parity.check(refs[-1], *got, where=f"hp={hp}")


def test_wide_exponent_gradients_every_element():
    """Replicas spanning many binades with cancellation: the fixed-order sum must
    still round like the exact one."""
    _need_gpu()
    rng = np.random.default_rng(5)
    n, S = 16, 30_000
    wl = _small_workload(n, S, rank=0)

    def bits(r):
        mant = rng.integers(0, 128, S)
        exp = rng.integers(-40, 8, S) + 127
        sign = rng.integers(0, 2, S)
        return ((sign << 15) | (exp << 7) | mant).astype(np.uint16)

    g_host = [np.concatenate([bits(r), np.zeros(wl.numel - S, np.uint16)]) for r in range(n)]
    master, m, v = parity.states_host(wl, np.arange(S))
    refs = oracle_trajectory(wl, np.arange(S), 1, 1, grads_fn=lambda r, t: g_host[r][:S],
                             init=(master, m, v))
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    dp.reduce_adam([to_dev_grad(g) for g in g_host], 0, S, dm, dmm, dv, dout, step=1, **HP)
    dp.stream_status()
    st = parity.check(refs[0], f32(dm), f32(dmm), f32(dv), u16(dout), where="wide exponents")
    assert st.bitwise_master > 0.999


# ---------------------------------------------------------------------------
# entry points, buckets, shards: bitwise invariances
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 13, 16])
def test_bucket_entries_match_full_buffer_bitwise(n):
    """Bucket sizes move elements between the vector body (scalar or packed
    lanes) and the scalar tail path; every split must give the same bits."""
    _need_gpu()
    wl = _small_workload(n, 50_021, rank=2)
    ref = _run_small_full(wl, entry="full")
    for entry, bucket in (("full", 1), ("full", 4096), ("bucket", 7), ("bucket", 4096),
                          ("buckets", 3), ("buckets", 1000), ("buckets", 50_021)):
        got = _run_small_full(wl, entry=entry, bucket=bucket)
        for a, b in zip(ref, got):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (entry, bucket)


def test_zero_shards_equal_the_data_parallel_update_bitwise():
    """Updating every rank's shard and concatenating equals one update of the
    whole flattened vector (ZeRO keeps data-parallel semantics)."""
    _need_gpu()
    n, S = 4, 10_007
    numel = n * S
    rng = np.random.default_rng(9)
    gh = [((rng.standard_normal(numel) * 1e-3).astype(np.float32)) for _ in range(n)]
    gh = [oracle.f32_to_bf16(g) for g in gh]
    th0 = (rng.standard_normal(numel) * 0.02).astype(np.float32)
    grads = [to_dev_grad(g) for g in gh]
    full = [torch.from_numpy(th0.copy()).cuda(), torch.zeros(numel, device="cuda"),
            torch.zeros(numel, device="cuda"), torch.empty(numel, dtype=torch.bfloat16,
                                                           device="cuda")]
    dp.reduce_adam_bucket(grads, 0, *full, step=1, **HP)
    parts = []
    for r in range(n):
        st = [torch.from_numpy(th0[r * S:(r + 1) * S].copy()).cuda(), torch.zeros(S, device="cuda"),
              torch.zeros(S, device="cuda"), torch.empty(S, dtype=torch.bfloat16, device="cuda")]
        dp.reduce_adam(grads, r, 1000, *st, step=1, **HP)
        parts.append(st)
    dp.stream_status()
    for k in range(4):
        cat = torch.cat([p[k] for p in parts])
        assert torch.equal(cat.view(torch.int16 if k == 3 else torch.int32),
                           full[k].view(torch.int16 if k == 3 else torch.int32))


def test_runs_are_bitwise_deterministic():
    _need_gpu()
    wl = _small_workload(8, 200_003, rank=5)
    a = _run_small_full(wl, steps=(1, 2, 3))
    b = _run_small_full(wl, steps=(1, 2, 3))
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_resume_from_saved_state_is_bitwise_identical():
    _need_gpu()
    wl = _small_workload(2, 30_000, rank=1)
    S = wl.shard_elems
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))

    def run(ts, st):
        dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in st)
        dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        for t in ts:
            grads = [to_dev_grad(g) for g in _host_full_buffers(wl, t)]
            dp.reduce_adam(grads, wl.shard_rank, S, dm, dmm, dv, dout, step=t, **HP)
        dp.stream_status()
        return f32(dm), f32(dmm), f32(dv), u16(dout)

    straight = run((1, 2, 3, 4), (master, m, v))
    half = run((1, 2), (master, m, v))
    resumed = run((3, 4), half[:3])   # "checkpoint": the states copied out and back in
    for x, y in zip(straight, resumed):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


@pytest.mark.parametrize("shift", [1, 3, 5, 7])
def test_unaligned_pointers_take_the_scalar_path_correctly(shift):
    _need_gpu()
    n, S = 3, 5_003
    wl = _small_workload(n, S, rank=0)
    gh = _host_full_buffers(wl, 1)
    master, m, v = parity.states_host(wl, np.arange(S))
    refs = oracle_trajectory(wl, np.arange(S), 1, 1, init=(master, m, v))
    # every buffer starts `shift` elements into a larger allocation
    grads = []
    for g in gh:
        big = torch.zeros(wl.numel + 8, dtype=torch.bfloat16, device="cuda")
        big[shift:shift + wl.numel] = to_dev_grad(g)
        grads.append(big[shift:shift + wl.numel])
    st = []
    for x in (master, m, v):
        big = torch.zeros(S + 8, device="cuda")
        big[shift:shift + S] = torch.from_numpy(x)
        st.append(big[shift:shift + S])
    bo = torch.zeros(S + 8, dtype=torch.bfloat16, device="cuda")
    dout = bo[shift:shift + S]
    dp.reduce_adam(grads, 0, S, st[0], st[1], st[2], dout, step=1, **HP)
    dp.stream_status()
    parity.check(refs[0], f32(st[0]), f32(st[1]), f32(st[2]), u16(dout), where=f"shift {shift}")


def test_outputs_outside_the_range_are_untouched():
    """Canaries around every state/output range survive a step."""
    _need_gpu()
    n, S, pad = 4, 33_333, 4096
    wl = _small_workload(n, S, rank=1)
    grads = [to_dev_grad(g) for g in _host_full_buffers(wl, 1)]
    canary = 12345.678
    bufs = [torch.full((S + 2 * pad,), canary, device="cuda") for _ in range(3)]
    bo = torch.full((S + 2 * pad,), canary, dtype=torch.bfloat16, device="cuda")
    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    for b, x in zip(bufs, (master, m, v)):
        b[pad:pad + S] = torch.from_numpy(x)
    views = [b[pad:pad + S] for b in bufs] + [bo[pad:pad + S]]
    dp.reduce_adam(grads, 1, 1000, *views, step=1, **HP)
    dp.stream_status()
    for b in bufs + [bo]:
        assert torch.all(b[:pad] == b.new_tensor(canary)) and torch.all(b[pad + S:] == b.new_tensor(canary))


def test_nonfinite_values_propagate_like_the_oracle():
    _need_gpu()
    n, S = 3, 4096
    wl = _small_workload(n, S, rank=0)
    gh = _host_full_buffers(wl, 1)
    master, m, v = parity.states_host(wl, np.arange(S))
    inf16, ninf16, nan16 = 0x7F80, 0xFF80, 0x7FC0
    gh[0][0:8] = inf16
    gh[1][8:16] = ninf16
    gh[0][16:24], gh[2][16:24] = inf16, ninf16
    gh[2][24:32] = nan16
    big = np.uint16(0x7F00)  # 2^127 + 2^127 overflows binary32: the average is +Inf
    gh[0][32:40] = big
    gh[1][32:40] = big
    master[40:48] = np.inf
    master[48:56] = np.nan
    m[56:64] = np.inf
    v[64:72] = np.inf
    refs = oracle_trajectory(wl, np.arange(S), 1, 1, grads_fn=lambda r, t: gh[r][:S],
                             init=(master.copy(), m.copy(), v.copy()))
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    dp.reduce_adam([to_dev_grad(g) for g in gh], 0, S, dm, dmm, dv, dout, step=1, **HP)
    dp.stream_status()
    parity.check(refs[0], f32(dm), f32(dmm), f32(dv), u16(dout), where="non-finite")


def test_empty_shard_and_zero_length_bucket_are_no_ops():
    _need_gpu()
    x = torch.zeros(4, device="cuda")
    o = torch.zeros(4, dtype=torch.bfloat16, device="cuda")
    g = torch.zeros(0, dtype=torch.bfloat16, device="cuda")
    dp.reduce_adam([g, g], 0, 1, x, x.clone(), x.clone(), o, step=1, **HP)
    dp.reduce_adam_bucket([g, g], 0, x, x.clone(), x.clone(), o, step=1, **HP)
    dp.stream_status()
    assert not x.any()


# ---------------------------------------------------------------------------
# full-size workloads: sampled elements
# ---------------------------------------------------------------------------

def _sample(S, bucket, rng, k=60_000):
    pts = [np.arange(min(S, 2048)), np.arange(max(0, S - 2048), S)]
    for b in range(bucket, S, bucket):
        pts.append(np.arange(max(0, b - 64), min(S, b + 64)))
    pts.append(rng.integers(0, S, size=k))
    return np.unique(np.concatenate(pts)).astype(np.int64)


def _free_bytes() -> int:
    """Device memory free for a new workload: what the driver reports plus what
    torch's caching allocator holds without using it (released first)."""
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    return free


def _fits(wl) -> bool:
    return workload_bytes(wl) + (4 << 30) < _free_bytes()


def _run_full_size(wl, entry):
    """The workload at its full size, sampled elements checked after every
    measured step: against the oracle's trajectory, and step by step from the
    GPU's own previous states.  entry: "full" (full replica buffers), "buckets"
    (the parameter-space bucket table) or "table" (every bucket in one launch)."""
    _need_gpu()
    if not _fits(wl):
        pytest.skip(f"{wl.name} needs {workload_bytes(wl) / 1e9:.1f} GB of device memory, "
                    f"{_free_bytes() / 1e9:.1f} GB free (4 GB kept back)")
    rng = np.random.default_rng(wl.seed)
    idx = _sample(wl.shard_elems, wl.bucket_elems, rng)
    t1 = wl.warmup_steps + wl.steps
    refs = oracle_trajectory(wl, idx, 1, t1)
    dev = DeviceWorkload(wl)
    dev.fill_states()
    tidx = torch.from_numpy(idx).cuda()
    stats = []
    if entry != "full":
        bs = dev.bucket_slices()
        table = (torch.empty(dp.bucket_table_bytes(wl.n_replicas, len(bs)), dtype=torch.uint8,
                             device="cuda") if entry == "table" else None)
        call = dp.BucketStep([s for _, s in bs], [o for o, _ in bs], dev.master, dev.m, dev.v,
                             dev.out, table)
    for t in range(1, t1 + 1):
        prev = (f32(dev.master[tidx]), f32(dev.m[tidx]), f32(dev.v[tidx]))
        dev.fill_grads(t)
        hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=t)
        launches = dp.dpopt_launch_count()
        if entry == "full":
            dp.reduce_adam(dev.grads, wl.shard_rank, wl.bucket_elems, dev.master, dev.m, dev.v,
                           dev.out, **hp)
        else:
            call.step(**hp)
        if entry == "table":
            assert dp.dpopt_launch_count() - launches == 1
        dp.stream_status()
        got = (f32(dev.master[tidx]), f32(dev.m[tidx]), f32(dev.v[tidx]), u16(dev.out[tidx]))
        parity.check_step(wl, idx, t, prev, got, wl.name)
        if t > wl.warmup_steps:
            stats.append(parity.check(refs[t - 1], *got, where=f"{wl.name} t={t}"))
    del dev, tidx
    if entry != "full":
        del bs, table, call
    _free_bytes()
    return stats


def test_gpt2_small_sized_buffer_sampled_ten_steps():
    st = _run_full_size(synth.WORKLOADS["gpt2s"], "full")
    assert min(s.bitwise_master for s in st) > 0.999


def test_1p3b_buffer_rank3_sampled_prewarmed():
    st = _run_full_size(synth.WORKLOADS["1p3b"], "full")
    assert min(s.bitwise_master for s in st) > 0.999


def test_70b_shard_n64_bucket_slices_sampled():
    """The 70B model's 1/64 shard as the benchmark runs it: 274 buckets of 64
    slices, every bucket in one launch."""
    st = _run_full_size(synth.WORKLOADS["70b_shard"], "table")
    assert min(s.bitwise_master for s in st) > 0.999


@pytest.mark.parametrize("S", [1_000_000, 16_000_000])
@pytest.mark.parametrize("n", synth.SWEEP_REPLICAS)
@pytest.mark.parametrize("kind", [0, 1])
def test_sweep_cells_sampled(S, n, kind):
    wl = synth.sweep_cell(S, n, kind)
    _run_full_size(wl, "buckets")


@pytest.mark.parametrize("S", [256_000_000, 1_000_000_000])
@pytest.mark.parametrize("n", synth.SWEEP_REPLICAS)
@pytest.mark.parametrize("kind", [0, 1])
def test_sweep_large_cells_sampled(S, n, kind):
    """Every cell of the sweep at 256M and 1B that fits the device: fp32
    replicas of 1e9 elements are 4 GB each, so byte offsets pass 2^32.  A cell
    that does not fit (fp32 x 64 x 1B needs 272 GB) is skipped with its size."""
    _run_full_size(synth.sweep_cell(S, n, kind), "buckets")
