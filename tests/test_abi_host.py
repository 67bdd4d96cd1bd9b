"""The C ABI on the host (no GPU): the library loads, exports every function
the header declares, and rejects bad arguments before touching the device."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

import oracle
from tests.test_oracle_pins import _golden_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dpopt.h")


@pytest.fixture(scope="module")
def dp():
    import __graft_entry__
    __graft_entry__.build_module().build()
    import zero_mixed_precision_gb300 as mod
    return mod


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dpopt_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(dp):
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(dp.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(dp.EXPORTED) == names


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles_standalone(lang, tmp_path):
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "dpopt.h"\nint main(void){return dpopt_status_string(0) == 0;}\n')
    cc = "gcc" if lang == "c" else "g++"
    subprocess.run([cc, "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-fsyntax-only",
                    str(src)], check=True)


def test_status_strings(dp):
    for code, name in ((0, "DPOPT_OK"), (1, "DPOPT_ERR_INVALID_ARG"), (2, "DPOPT_ERR_UNSUPPORTED"),
                       (3, "DPOPT_ERR_CUDA"), (4, "DPOPT_ERR_TIMEOUT"), (5, "DPOPT_ERR_BOUNDS"),
                       (99, "DPOPT_UNKNOWN_STATUS")):
        assert dp.dpopt_status_string(code) == name


def test_bounds_checked_build_exports_the_same_interface(dp):
    """The bounds-checked variant is the same interface: every declared symbol,
    the same status strings, a version marked "+bounds"; the release build
    refuses the bounds self-test (it has no checks)."""
    lib = ctypes.CDLL(dp.binding._build.lib_path("bounds"))
    for n in _declared():
        assert hasattr(lib, n), n
    lib.dpopt_version.restype = ctypes.c_char_p
    lib.dpopt_status_string.restype = ctypes.c_char_p
    assert lib.dpopt_version().decode().endswith("+bounds")
    assert lib.dpopt_status_string(5).decode() == "DPOPT_ERR_BOUNDS"
    assert not dp.dpopt_version().endswith("+bounds")
    assert dp.dpopt_selftest_bounds(0) == dp.DPOPT_ERR_UNSUPPORTED


@pytest.mark.parametrize("row", [r for r in _golden_rows() if r[4] == "total"],
                         ids=lambda r: r[7][:40])
def test_state_bytes_matches_printed_figures(dp, row):
    psi, variant, n_dp, stage, _comp, expected, rel, _cite = row
    rc, got = dp.dpopt_state_bytes(int(psi), variant, n_dp, stage)
    assert rc == 0
    if rel == "eq":
        assert got == pytest.approx(expected, rel=1e-12)
    elif rel == "r1":   # printed to one decimal of a GB
        assert round(got / 1e8) == round(expected / 1e8), (got, expected)
    else:
        assert got > expected


@pytest.mark.parametrize("variant", [0, 1])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("n_dp", [1, 8, 64])
def test_state_bytes_agrees_with_the_oracle_accounting(dp, variant, stage, n_dp):
    rc, got = dp.dpopt_state_bytes(70_000_000_000, variant, n_dp, stage)
    assert rc == 0 and got == pytest.approx(oracle.state_bytes(70e9, variant, n_dp, stage), rel=1e-12)


def test_state_bytes_rejects_bad_arguments(dp):
    for args in ((-1, 0, 1, 0), (1, 2, 1, 0), (1, 0, 0, 0), (1, 0, 1, 4)):
        assert dp.dpopt_state_bytes(*args)[0] == dp.DPOPT_ERR_INVALID_ARG


@pytest.mark.parametrize("shard,bucket", [(0, 5), (1, 1), (10, 3), (31_000_000, 25_000_000),
                                          (162_500_000, 50_000_000), (1_093_750_000, 4_000_000),
                                          (7, 100)])
def test_bucket_iterator_agrees_with_the_oracle_ranges(dp, shard, bucket):
    want = oracle.bucket_ranges(shard, bucket)
    rc, cnt = dp.dpopt_bucket_count(shard, bucket)
    assert rc == 0 and cnt == len(want)
    for i, (off, ln) in enumerate(want):
        assert dp.dpopt_bucket_range(shard, bucket, i) == (0, off, ln)
    assert dp.dpopt_bucket_range(shard, bucket, cnt)[0] == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_bucket_range(shard, bucket, -1)[0] == dp.DPOPT_ERR_INVALID_ARG


def test_bucket_iterator_rejects_bad_arguments(dp):
    assert dp.dpopt_bucket_count(-1, 5)[0] == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_bucket_count(5, 0)[0] == dp.DPOPT_ERR_INVALID_ARG


# Fake, never-dereferenced device addresses: validation fails before any launch.
G = [0x10_0000_0000 + r * 0x1_0000_0000 for r in range(64)]
MASTER, M, V, OUT = 0x90_0000_0000, 0xA0_0000_0000, 0xB0_0000_0000, 0xC0_0000_0000
HP = (1e-3, 0.9, 0.999, 1e-8)


def _full(dp, **over):
    a = dict(grads=G[:4], n=4, numel=4096, rank=0, bucket=1024, master=MASTER, m=M, v=V, out=OUT,
             lr=HP[0], b1=HP[1], b2=HP[2], eps=HP[3], step=1, dtype=0)
    a.update(over)
    return dp.dpopt_reduce_adam_ex(a["grads"], a["dtype"], a["n"], a["numel"], a["rank"],
                                   a["bucket"], a["master"], a["m"], a["v"], a["out"], a["lr"],
                                   a["b1"], a["b2"], a["eps"], a["step"], 0)


@pytest.mark.parametrize("over,code", [
    (dict(n=0), 1), (dict(n=65, grads=G[:64] + [G[0]]), 2), (dict(numel=4095), 1),
    (dict(numel=-4), 1), (dict(rank=4), 1), (dict(rank=-1), 1), (dict(bucket=0), 1),
    (dict(step=0), 1), (dict(step=-3), 1), (dict(lr=float("nan")), 1), (dict(lr=float("inf")), 1),
    (dict(b1=1.0), 1), (dict(b1=-0.1), 1), (dict(b2=1.0), 1), (dict(b2=float("nan")), 1),
    (dict(eps=-1e-8), 1), (dict(eps=float("inf")), 1), (dict(master=0), 1), (dict(out=0), 1),
    (dict(grads=[G[0], 0, G[2], G[3]]), 1), (dict(dtype=7), 1), (dict(master=MASTER + 2), 1),
    (dict(out=OUT + 1), 1), (dict(grads=[G[0] + 1, G[1], G[2], G[3]]), 1),
    (dict(m=MASTER + 8), 1),                      # m overlaps master
    (dict(out=G[0] + 2), 1),                      # output inside gradient buffer 0's shard
    (dict(master=G[1] + 1000), 1),                # state inside a gradient shard
])
def test_full_buffer_entry_rejects_bad_arguments(dp, over, code):
    assert _full(dp, **over) == code
    assert dp.dpopt_last_error() != ""


def test_kernel_policy_round_trip_and_rejects_unknown(dp):
    assert dp.dpopt_get_kernel_policy() == dp.DPOPT_KERNEL_AUTO
    for pol in (dp.DPOPT_KERNEL_DIRECT, dp.DPOPT_KERNEL_BULK, dp.DPOPT_KERNEL_AUTO):
        assert dp.dpopt_set_kernel_policy(pol) == 0 and dp.dpopt_get_kernel_policy() == pol
    assert dp.dpopt_set_kernel_policy(7) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_get_kernel_policy() == dp.DPOPT_KERNEL_AUTO


def test_selftest_rejects_out_of_range_limits(dp):
    assert dp.dpopt_selftest_wait_timeout(0, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_selftest_wait_timeout(3_000_000_000, 0) == dp.DPOPT_ERR_INVALID_ARG


def test_null_grads_table_is_rejected(dp):
    assert dp.dpopt_reduce_adam(None, 2, 8, 0, 4, MASTER, M, V, OUT, *HP, 1, 0) == 1


def test_bucket_entries_reject_bad_arguments(dp):
    args = (MASTER, M, V, OUT, *HP, 1, 0)
    assert dp.dpopt_reduce_adam_bucket(G[:2], 0, 2, -1, 10, *args) == 1
    assert dp.dpopt_reduce_adam_bucket(G[:2], 0, 2, 0, -5, *args) == 1
    assert dp.dpopt_reduce_adam_bucket(G[:2], 3, 2, 0, 10, *args) == 1
    # overlapping buckets
    assert dp.dpopt_reduce_adam_buckets(G[:4], 0, 2, [0, 5], [10, 10], *args) == 1
    # a slice that overlaps the master range
    assert dp.dpopt_reduce_adam_buckets([G[0], MASTER + 16], 0, 2, [0], [100], *args) == 1
    # n_replicas beyond the limit
    assert dp.dpopt_reduce_adam_buckets(G[:64] * 2, 0, 65, [0], [10], *args) == 2


def test_bucket_average_norm_rejects_bad_arguments(dp):
    SQ, SCR, AVG = 0xD0_0000_0000, 0xE0_0000_0000, 0xC8_0000_0000
    L = 5000                                       # two buckets: 10000 elements, 3 chunks
    nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(2 * L, 2)[1]
    # two buckets continuing one another in the shard and in both replicas
    joined = [G[0], G[1], G[0] + 2 * L, G[1] + 2 * L]

    def call(table=joined, offs=(0, L), avg=AVG, scr=SCR, nb=nbytes):
        return dp.dpopt_grad_average_sqnorm_buckets(table, 0, 2, list(offs), [L, L], 0.0,
                                                    avg, SQ, scr, nb, 0)
    assert call(avg=0) == dp.DPOPT_ERR_INVALID_ARG
    assert call(avg=AVG + 2) == dp.DPOPT_ERR_INVALID_ARG
    assert call(avg=SCR - 4 * 1000) == dp.DPOPT_ERR_INVALID_ARG    # overlaps the partials
    assert call(avg=G[1] - 4 * 10) == dp.DPOPT_ERR_INVALID_ARG     # overlaps a gradient
    assert call(nb=16) == dp.DPOPT_ERR_INVALID_ARG                 # 3 partials needed
    # buckets that do not continue one another (a gap in replica 1's memory)
    apart = [G[0], G[1], G[0] + 2 * L, G[1] + 2 * L + 64]
    assert call(table=apart) == dp.DPOPT_ERR_UNSUPPORTED
    # ... or in the shard
    assert call(offs=(0, L + 16)) == dp.DPOPT_ERR_UNSUPPORTED
    # the loss-scaled form: its state pointer is checked first
    STATE = 0xF8_0000_0000

    def amp(state, avg=AVG):
        return dp.dpopt_amp_average_sqnorm_buckets(joined, 2, 2, [0, L], [L, L], state, avg, SQ,
                                                   SCR, nbytes, 0)
    assert amp(0) == dp.DPOPT_ERR_INVALID_ARG
    assert amp(STATE + 4) == dp.DPOPT_ERR_INVALID_ARG
    assert amp(STATE, avg=0) == dp.DPOPT_ERR_INVALID_ARG
    assert amp(STATE, avg=AVG + 1) == dp.DPOPT_ERR_INVALID_ARG
    # the readiness-driven form: events are required, buckets need not join
    def ready(events, table=joined):
        return dp.dpopt_grad_sqnorm_buckets_when_ready(table, 0, 2, [0, L], [L, L], events, 0.0,
                                                       AVG, SQ, SCR, nbytes, 0)
    assert ready(None) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_amp_sqnorm_buckets_when_ready(joined, 2, 2, [0, L], [L, L], [0, 0], 0, AVG,
                                                  SQ, SCR, nbytes, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_amp_sqnorm_buckets_when_ready(joined, 2, 2, [0, L], [L, L], None, STATE,
                                                  AVG, SQ, SCR, nbytes, 0) == \
        dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_grad_sqnorm_buckets_when_ready(joined, 0, 2, [0, L], [L, L], [0, 0], 0.0,
                                                   AVG + 2, SQ, SCR, nbytes, 0) == \
        dp.DPOPT_ERR_INVALID_ARG


def test_bucket_table_bytes(dp):
    # 274 buckets of 64 slices (a 70B model's 1/64 shard in 4M buckets)
    assert dp.dpopt_bucket_table_bytes(64, 274) == (0, 32 * 275 + 8 * 274 * 64)
    assert dp.dpopt_bucket_table_bytes(1, 0) == (0, 32)
    assert dp.dpopt_bucket_table_bytes(0, 1)[0] == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_bucket_table_bytes(65, 1)[0] == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_bucket_table_bytes(2, -1)[0] == dp.DPOPT_ERR_INVALID_ARG


def test_table_entry_rejects_bad_arguments(dp):
    TAB = 0xF0_0000_0000
    need = dp.dpopt_bucket_table_bytes(2, 2)[1]

    def call(table=TAB, nbytes=need, table_slices=G[:4], offs=(0, 10), lens=(10, 10), n=2,
             master=MASTER, opts=None, step=1):
        return dp.dpopt_reduce_adam_buckets_table(table_slices, 0, n, list(offs), list(lens),
                                                  master, M, V, OUT, *HP, step, opts, table,
                                                  nbytes, 0)
    assert call(table=0) == 1                    # no table
    assert call(table=TAB + 8) == 1              # not 16-byte aligned
    assert call(nbytes=need - 1) == 1            # too small
    assert call(table=MASTER) == 1               # the table overlaps the master range
    assert call(table=G[1] - 64) == 1            # a slice overlaps the table
    assert call(offs=(0, 5)) == 1                # overlapping buckets
    assert call(step=0) == 1
    assert call(n=65, table_slices=G[:64] * 3, offs=(0, 10), lens=(10, 10)) == 2
    assert call(opts=dp.StepOptions(-0.1, 0.0, None, 0.0)) == 1
    assert dp.dpopt_last_error() != ""


def test_sqnorm_scratch_bytes(dp):
    assert dp.dpopt_grad_sqnorm_scratch_bytes(0, 1) == (0, 8)
    assert dp.dpopt_grad_sqnorm_scratch_bytes(65536, 1) == (0, 8 * (65536 // 4096 + 1))
    assert dp.dpopt_grad_sqnorm_scratch_bytes(4097, 0) == (0, 16)
    assert dp.dpopt_grad_sqnorm_scratch_bytes(65537, 1) == (0, 8 * (17 + 1))
    assert dp.dpopt_grad_sqnorm_scratch_bytes(1_093_750_000, 274)[1] == 8 * (267_029 + 274)
    assert dp.dpopt_grad_sqnorm_scratch_bytes(-1, 1)[0] == dp.DPOPT_ERR_INVALID_ARG


def test_sqnorm_and_adamw_reject_bad_arguments(dp):
    SQ, SCR = 0xD0_0000_0000, 0xE0_0000_0000
    ok = dict(grads=G[:2], dt=0, n=2, numel=2 * 70000, rank=0, un=0.0, out=SQ, scr=SCR, nbytes=16)

    def call(**kw):
        a = dict(ok, **kw)
        return dp.dpopt_grad_sqnorm(a["grads"], a["dt"], a["n"], a["numel"], a["rank"], a["un"],
                                    a["out"], a["scr"], a["nbytes"], 0)
    assert call(out=0) == 1
    assert call(out=SQ + 4) == 1
    assert call(scr=0) == 1
    assert call(nbytes=8) == 1                   # 70000 elements need two partials
    assert call(un=-1.0) == 1
    assert call(un=float("nan")) == 1
    assert call(out=SCR + 8) == 1                # output inside the partials
    assert call(grads=[SQ - 16, G[1]]) == 1      # gradients overlap the output
    assert call(numel=7) == 1
    assert call(n=65, grads=G[:64] + [G[0]]) == 2
    AVG = 0xC0_0000_0000

    def call_avg(avg, **kw):
        a = dict(ok, **kw)
        return dp.dpopt_grad_average_sqnorm(a["grads"], a["dt"], a["n"], a["numel"], a["rank"],
                                            a["un"], avg, a["out"], a["scr"], a["nbytes"], 0)
    assert call_avg(0) == 1                      # no destination for the average
    assert call_avg(AVG + 2) == 1                # not 4-byte aligned
    assert call_avg(SCR - 16) == 1               # overlaps the partials
    assert call_avg(SQ - 64) == 1                # overlaps the norm output
    assert call_avg(G[0] - 8) == 1               # overlaps a gradient
    assert call_avg(AVG, nbytes=8) == 1          # the norm's own checks still apply
    opt = dp.StepOptions(-0.1, 0.0, None, 0.0)
    assert dp.dpopt_reduce_adamw(G[:4], 0, 4, 4096, 0, 1024, MASTER, M, V, OUT, *HP, 1, opt, 0) == 1
    opt = dp.StepOptions(0.01, 1.0, None, 0.0)   # clipping without a norm pointer
    assert dp.dpopt_reduce_adamw(G[:4], 0, 4, 4096, 0, 1024, MASTER, M, V, OUT, *HP, 1, opt, 0) == 1
    opt = dp.StepOptions(0.01, 1.0, SQ + 3, 0.0)  # misaligned norm pointer
    assert dp.dpopt_reduce_adamw(G[:4], 0, 4, 4096, 0, 1024, MASTER, M, V, OUT, *HP, 1, opt, 0) == 1
    # the loss-scaled step: its norm may be null only without clipping
    STATE = 0xF0_0000_0000
    cfg = dp.LossScaleConfig(1024.0, 10, 2, 1.0)

    def amp(sq, max_norm, lr_dev=0):
        return dp.dpopt_amp_step(G[:4], 0, 4, 4096, 0, 1024, MASTER, M, V, OUT, *HP, 0.01,
                                 max_norm, sq, STATE, cfg, lr_dev, 0)
    assert amp(0, 1.0) == 1
    assert amp(SQ + 4, 0.0) == 1
    assert amp(0, 0.0, lr_dev=0xF4_0000_0002) == 1      # a misaligned learning-rate pointer


def test_binding_refuses_pageable_host_operands(dp):
    """Pinned host memory is a valid operand (the kernels address it in place);
    pageable host memory is refused by the binding before any call into the
    library, for gradients, states and the output alike."""
    import torch
    S = 64
    g = [torch.zeros(S, dtype=torch.bfloat16) for _ in range(2)]
    st = [torch.zeros(S) for _ in range(3)]
    out = torch.zeros(S, dtype=torch.bfloat16)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=1, stream=0)
    with pytest.raises(ValueError, match="pageable"):
        dp.reduce_adam_bucket(g, 0, *st, out, **hp)
    with pytest.raises(ValueError, match="pageable"):
        dp.reduce_adam(g, 0, S, *st, out, **hp)


# replica parameter buffers of the fused step + all-gather (fake addresses)
R = [0xD0_0000_0000 + r * 0x1_0000_0000 for r in range(64)]


def _fused(dp, **over):
    a = dict(grads=G[:4], n=4, numel=4096, rank=1, bucket=1024, master=MASTER, m=M, v=V,
             reps=R[:4], lr=HP[0], b1=HP[1], b2=HP[2], eps=HP[3], step=1, dtype=0)
    a.update(over)
    return dp.dpopt_reduce_adam_allgather(a["grads"], a["dtype"], a["n"], a["numel"], a["rank"],
                                          a["bucket"], a["master"], a["m"], a["v"], a["reps"],
                                          a["lr"], a["b1"], a["b2"], a["eps"], a["step"], 0)


@pytest.mark.parametrize("over,code", [
    (dict(reps=None), 1), (dict(reps=[R[0], 0, R[2], R[3]]), 1),
    (dict(reps=[R[0], R[1] + 1, R[2], R[3]]), 1),          # misaligned replica buffer
    (dict(reps=[R[0], R[1], R[1] + 1000, R[3]]), 1),      # two destinations overlap
    (dict(reps=[R[0], R[1], MASTER - 1024 * 2 + 16, R[3]]), 1),  # a destination on master
    (dict(reps=[R[0], R[1], G[0], R[3]]), 1),             # a destination on a gradient shard
    (dict(master=R[1] + 2048 + 64), 1),                   # master on the working copy
    (dict(rank=4), 1), (dict(rank=-1), 1), (dict(numel=4095), 1), (dict(step=0), 1),
    (dict(n=65, grads=G[:64] + [G[0]], reps=R[:64] + [R[0]]), 2), (dict(dtype=5), 1),
    (dict(b1=1.0), 1), (dict(bucket=0), 1), (dict(grads=None), 1),
])
def test_fused_allgather_entry_rejects_bad_arguments(dp, over, code):
    assert _fused(dp, **over) == code
    assert dp.dpopt_last_error() != ""


def test_fused_allgather_entry_with_nothing_to_update_checks_and_returns(dp):
    assert _fused(dp, numel=0) == 0
    assert _fused(dp, numel=0, rank=7) == 1


def test_gather_policy_round_trip_and_rejects_unknown(dp):
    assert dp.dpopt_get_gather_policy() == dp.DPOPT_GATHER_AUTO
    for pol in (dp.DPOPT_GATHER_FUSED, dp.DPOPT_GATHER_SEPARATE, dp.DPOPT_GATHER_AUTO):
        assert dp.dpopt_set_gather_policy(pol) == 0 and dp.dpopt_get_gather_policy() == pol
    assert dp.dpopt_set_gather_policy(3) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_get_gather_policy() == dp.DPOPT_GATHER_AUTO
