"""A battery of library calls that walks every kernel's index paths: full
buffers and batched buckets with ragged tails, unaligned slices (the
one-element path), the bulk-copy kernel, the runtime-replica-count kernels
(unrolled in three batches at N = 18, the shared-memory walk at N = 24 and
40, the register walk at N = 64),
the one-launch bucket entry (launch table in device memory, and contiguous
buckets joined), the norm pre-pass with and without the stored average (over
full buffers, over joined buckets, and bucket by bucket as each is ready), the
loss-scaled step, the all-gather and the fused step + all-gather (per-thread
stores, and whole tiles written by bulk copies).

run() returns every output as numpy arrays plus the stream status after each
call.  tests/test_gpu_bounds.py runs it once on the release library in the
test process and once, in a child process started with
DPOPT_LIB_VARIANT=bounds, on the bounds-checked build, and compares the two.
Run as a script: python -m tests.bounds_battery OUT.npz
"""
from __future__ import annotations

import sys

import numpy as np
import torch

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _rand(gen, n, scale, dtype):
    return (torch.randn(n, generator=gen, device="cuda") * scale).to(dtype)


def _states(gen, S):
    return [torch.randn(S, generator=gen, device="cuda") * 0.02,
            torch.randn(S, generator=gen, device="cuda") * 1e-4,
            (torch.randn(S, generator=gen, device="cuda") * 1e-6).abs()]


def _host(t: torch.Tensor) -> np.ndarray:
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().copy()
    return t.cpu().numpy().copy()


def run() -> tuple[dict, list]:
    import zero_mixed_precision_gb300 as dp

    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    out: dict[str, np.ndarray] = {}
    status: list[tuple[str, int]] = []

    def keep(name, *tensors):
        torch.cuda.synchronize()
        status.append((name, dp.dpopt_stream_status(0)))
        for i, t in enumerate(tensors):
            out[f"{name}/{i}"] = _host(t)

    # full-buffer step: unrolled N, the runtime-count kernel, bf16 / fp32 / fp16
    for n, S, dt in ((1, 10_007, torch.bfloat16), (2, 9_001, torch.bfloat16),
                     (3, 8_195, torch.bfloat16), (4, 12_289, torch.bfloat16),
                     (8, 4_099, torch.bfloat16), (13, 3_001, torch.bfloat16),
                     (18, 2_011, torch.bfloat16), (24, 2_003, torch.bfloat16),
                     (40, 1_001, torch.float16),
                     (2, 7_003, torch.float32), (3, 5_005, torch.float32),
                     (5, 6_007, torch.float32), (4, 4_103, torch.float16)):
        rank = n // 2
        grads = [_rand(gen, n * S, 1e-3, dt) for _ in range(n)]
        st = _states(gen, S)
        o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        dp.reduce_adam(grads, rank, 1000, *st, o, step=3, **HP)
        keep(f"full_n{n}_{str(dt)[6:]}", *st, o)

    # the bulk-copy kernel where it applies
    with dp.kernel_policy(dp.DPOPT_KERNEL_BULK):
        n, S = 4, 20_011
        grads = [_rand(gen, n * S, 1e-3, torch.bfloat16) for _ in range(n)]
        st = _states(gen, S)
        o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        dp.reduce_adam(grads, 1, S, *st, o, step=2, **HP)
        keep("bulk_n4", *st, o)

    # batched buckets: ragged lengths, unaligned offsets, more buckets than one
    # launch's table holds at N = 64 (several launches)
    for n, lens in ((4, [1, 7, 8, 15, 4097, 1000, 33, 2]), (64, [37] * 40 + [5])):
        S = sum(lens)
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
        slices = [[_rand(gen, ln, 1e-3, torch.bfloat16) for _ in range(n)] for ln in lens]
        st = _states(gen, S)
        o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        dp.reduce_adam_buckets(slices, offs, *st, o, step=4, **HP)
        keep(f"buckets_n{n}", *st, o)
        st2 = _states(gen, S)
        o2 = torch.empty(S, dtype=torch.bfloat16, device="cuda")
        dp.reduce_adam_buckets_when_ready(slices[::-1], offs[::-1], [None] * len(lens), *st2, o2,
                                          step=4, **HP)
        keep(f"when_ready_n{n}", *st2, o2)

    # every bucket in one launch: separate slices through a launch table in
    # device memory, and contiguous slices joined into one segment
    n = 8
    lens = [37, 8, 4096, 1, 2048] * 40 + [5]
    S = sum(lens)
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
    slices = [[_rand(gen, ln, 1e-3, torch.bfloat16) for _ in range(n)] for ln in lens]
    table = torch.empty(dp.bucket_table_bytes(n, len(lens)), dtype=torch.uint8, device="cuda")
    st = _states(gen, S)
    o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    dp.reduce_adam_buckets_table(slices, offs, *st, o, table, step=3, **HP)
    keep("table_n8", *st, o)
    flat = [_rand(gen, S, 1e-3, torch.bfloat16) for _ in range(n)]
    rows = [[f[off:off + ln] for f in flat] for off, ln in zip(offs, lens)]
    st = _states(gen, S)
    dp.reduce_adam_buckets(rows, offs, *st, o, step=3, **HP)
    keep("joined_n8", *st, o)

    # unaligned slices: every pointer one element past an aligned address
    n, S = 3, 6_001
    bufs = [_rand(gen, S + 1, 1e-3, torch.bfloat16) for _ in range(n)]
    st = [x for x in _states(gen, S + 1)]
    o = torch.empty(S + 1, dtype=torch.bfloat16, device="cuda")
    dp.reduce_adam_bucket([b[1:] for b in bufs], 1, *st, o, step=1, **HP)
    keep("unaligned", *st, o)

    # norm pre-pass: full buffer, stored average, buckets, built-in scratch
    n, S = 4, 30_001
    grads = [_rand(gen, n * S, 1e-3, torch.bfloat16) for _ in range(n)]
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)[1] // 8 + 1,
                          dtype=torch.float64, device="cuda")
    dp.grad_sqnorm(grads, 2, sq, scratch)
    keep("sqnorm", sq)
    avg = torch.empty(S, device="cuda")
    sq2 = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_average_sqnorm(grads, 2, avg, sq2, scratch)
    keep("average_sqnorm", avg, sq2)
    sq3 = torch.zeros(1, dtype=torch.float64, device="cuda")
    lens = [4097, 1, 9000, 333]
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
    slices = [[_rand(gen, ln, 1e-3, torch.bfloat16) for _ in range(n)] for ln in lens]
    sc = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(sum(lens), len(lens))[1] // 8 + 1,
                     dtype=torch.float64, device="cuda")
    dp.grad_sqnorm_buckets(slices, offs, sq3, sc)
    keep("sqnorm_buckets", sq3)
    # the same lengths as consecutive views of flat buffers: joined into one
    # segment, the average stored at each element's shard offset
    flat = [_rand(gen, sum(lens), 1e-3, torch.bfloat16) for _ in range(n)]
    joined = [[f[o:o + ln] for f in flat] for o, ln in zip(offs, lens)]
    avg_b = torch.full((sum(lens) + 8,), float("nan"), device="cuda")
    sq5 = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_average_sqnorm_buckets(joined, offs, avg_b[:sum(lens)], sq5, sc)
    keep("average_sqnorm_buckets", avg_b, sq5)
    # bucket by bucket as each is ready (here: listed last first, null events),
    # the separate slices, the average stored for each
    avg_r = torch.full((sum(lens) + 8,), float("nan"), device="cuda")
    sq6 = torch.zeros(1, dtype=torch.float64, device="cuda")
    dp.grad_sqnorm_buckets_when_ready(slices[::-1], offs[::-1], [None] * len(lens), sq6, sc,
                                      avg_out=avg_r[:sum(lens)])
    keep("sqnorm_buckets_when_ready", avg_r, sq6)
    sq4 = torch.zeros(1, dtype=torch.float64, device="cuda")
    rc = dp.dpopt_grad_sqnorm_noalloc([g.data_ptr() for g in grads], dp.DPOPT_GRAD_BF16, n,
                                      n * S, 2, 0.0, sq4.data_ptr(), 0)
    assert rc == 0
    keep("sqnorm_noalloc", sq4)

    # clipped AdamW through the stored average, and the fused form
    st = _states(gen, S)
    o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    opts = dp.step_options(weight_decay=0.01, max_grad_norm=1e-3, grad_sqnorm=sq2)
    dp.reduce_adamw([avg], 0, S, *st, o, step=5, opts=opts, **HP)
    keep("adamw_stored", *st, o)
    st = _states(gen, S)
    dp.reduce_adamw(grads, 2, 4096, *st, o, step=5, opts=opts, **HP)
    keep("adamw_fused", *st, o)

    # loss-scaled fp16 steps (one with an overflow)
    n, S = 2, 8_191
    state = torch.zeros(4, dtype=torch.int64, device="cuda")
    cfg = dp.loss_scale_init(state, init_scale=1024.0, window=2, hysteresis=1)
    st = _states(gen, S)
    o = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    sc = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)[1] // 8 + 1, dtype=torch.float64,
                     device="cuda")
    for it in range(3):
        grads = [_rand(gen, n * S, 1.0, torch.float16) for _ in range(n)]
        if it == 1:
            grads[0][5] = float("inf")
        sqn = torch.zeros(1, dtype=torch.float64, device="cuda")
        dp.amp_sqnorm(grads, 1, state, sqn, sc)
        dp.amp_step(grads, 1, 1000, *st, o, weight_decay=0.01, max_grad_norm=1.0,
                    global_sqnorm=sqn, state=state, cfg=cfg, **HP)
        keep(f"amp_{it}", *st, o, state)

    # all-gather, and the step fused with it (aligned and unaligned replicas)
    n, S, rank = 4, 9_999, 3
    shard = _rand(gen, S, 1.0, torch.bfloat16)
    reps = [torch.zeros(n * S, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    dp.allgather_bf16(shard, rank, reps)
    keep("allgather", *reps)
    grads = [_rand(gen, n * S, 1e-3, torch.bfloat16) for _ in range(n)]
    for tag, off in (("aligned", 0), ("unaligned", 1)):
        base = [torch.zeros(n * S + 8, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        reps = [b[off:off + n * S] for b in base]
        st = _states(gen, S)
        dp.reduce_adam_allgather(grads, rank, 2048, *st, reps, step=2, **HP)
        keep(f"fused_gather_{tag}", *st, *base)
    # a shard whose replica ranges are 16-byte aligned: whole 2048-element tiles
    # go out as bulk copies, the last group by per-thread stores
    n, S, rank = 4, 20_488, 3
    grads = [_rand(gen, n * S, 1e-3, torch.bfloat16) for _ in range(n)]
    reps = [torch.zeros(n * S, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    st = _states(gen, S)
    dp.reduce_adam_allgather(grads, rank, 2048, *st, reps, step=2, **HP)
    keep("fused_gather_tiles", *st, *reps)
    return out, status


def selftest() -> list[int]:
    """The deliberate check failure: reported once, then cleared."""
    import zero_mixed_precision_gb300 as dp
    return [dp.dpopt_selftest_bounds(0), dp.dpopt_stream_status(0), dp.dpopt_stream_status(0)]


def main(path: str) -> None:
    import zero_mixed_precision_gb300 as dp
    torch.cuda.set_device(0)
    out, status = run()
    st = selftest()
    np.savez(path, **out, __status__=np.array([s for _, s in status]),
             __names__=np.array([nm for nm, _ in status]), __selftest__=np.array(st),
             __version__=np.array(dp.dpopt_version()))


if __name__ == "__main__":
    main(sys.argv[1])
