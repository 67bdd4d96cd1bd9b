"""Pins of the CPU oracle against things other than itself.

Each test ties one part of the oracle to a fact fixed outside it: a figure
printed on the pages (tests/golden/), a closed form, a brute-force exact
computation with rationals, an invariant, or a library routine (torch CPU
bf16 rounding, torch.optim.Adam / AdamW in float64).  They are chosen so
that a dropped term, a wrong sign or index, or swapped operands in the
oracle fail at least one of them (see test_planted_mistakes_are_caught).
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

U = 2.0 ** -24  # unit roundoff of binary32
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# exact-rational helpers (independent of the oracle)
# ---------------------------------------------------------------------------

def frac_to_f32(q: Fraction) -> float:
    """Round an exact rational to the nearest binary32, ties to even."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    qexp = max(e, -126) - 23          # spacing of binary32 numbers around a
    scaled = a / Fraction(2) ** qexp
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = Fraction(n) * Fraction(2) ** qexp
    if val >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * float(val)


def bits_to_frac_bf16(h: int) -> Fraction:
    f = np.array([h << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def rand_bf16(rng, shape, lo_exp=-30, hi_exp=10):
    """Random finite bf16 bit patterns with exponents spread over [lo_exp, hi_exp)."""
    mant = rng.integers(0, 128, size=shape)
    exp = rng.integers(lo_exp, hi_exp, size=shape) + 127
    sign = rng.integers(0, 2, size=shape)
    return ((sign << 15) | (exp << 7) | mant).astype(np.uint16)


# ---------------------------------------------------------------------------
# bf16 encoding
# ---------------------------------------------------------------------------

def test_bf16_rne_matches_torch_cpu_library_rounding():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, 3.4028235e38,
                         1e-40, -1e-40, 1.401298464e-45, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                         1.0 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    # exact ties on both parities of the kept last bit
    ties = (np.arange(0, 4096, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, specials, ties[np.isfinite(ties)]])
    ours = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_nan_stays_quiet_nan():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    x = np.concatenate([x, np.array([0x7F800001, 0xFF800001, 0x7FC00000], dtype=np.uint32)
                        .view(np.float32)])
    out = oracle.f32_to_bf16(x)
    widened = oracle.bf16_to_f64(out)
    assert np.all(np.isnan(widened))
    assert np.all(out & 0x0040)


def test_bf16_widening_is_exact_like_torch():
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])
    assert np.all(np.isnan(ours[np.isnan(ref)]))
    assert np.all(ours[np.isinf(ref)] == ref[np.isinf(ref)])


# ---------------------------------------------------------------------------
# the reduce half: fixed-order average
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8])
def test_average_equals_exact_rational_average_bruteforce(n):
    """g = fl32(fl32(sum)/N) with the sum exact: brute force with Fractions."""
    rng = np.random.default_rng(100 + n)
    count = 512
    grads = [rand_bf16(rng, count) for _ in range(n)]
    got = oracle.average(grads)
    for j in range(count):
        s = sum(bits_to_frac_bf16(int(g[j])) for g in grads)
        s32 = frac_to_f32(s)
        want = frac_to_f32(Fraction(s32) / n)
        assert got[j] == np.float32(want), (j, got[j], want)


def test_average_fp32_grads_bruteforce():
    rng = np.random.default_rng(7)
    n, count = 5, 400
    grads = [(rng.standard_normal(count) * 10.0 ** rng.integers(-6, 3, count))
             .astype(np.float32) for _ in range(n)]
    got = oracle.average(grads)
    for j in range(count):
        s = sum(Fraction(float(g[j])) for g in grads)
        want = frac_to_f32(Fraction(frac_to_f32(s)) / n)
        assert got[j] == np.float32(want)


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 13, 32, 64])
def test_identical_replicas_average_to_the_input_exactly(n):
    rng = np.random.default_rng(n)
    x = rand_bf16(rng, 4096, lo_exp=-120, hi_exp=100)
    got = oracle.average([x] * n)
    np.testing.assert_array_equal(got.view(np.uint32), (x.astype(np.uint32) << 16))


def test_single_replica_is_identity():
    rng = np.random.default_rng(3)
    x = rand_bf16(rng, 1000)
    np.testing.assert_array_equal(oracle.average([x]), oracle.bf16_to_f64(x).astype(np.float32))


def test_permuting_replicas_leaves_average_unchanged():
    rng = np.random.default_rng(4)
    grads = [rand_bf16(rng, 2048, lo_exp=-20, hi_exp=5) for _ in range(8)]
    a = oracle.average(grads)
    for perm in ([7, 6, 5, 4, 3, 2, 1, 0], [3, 1, 4, 0, 5, 2, 7, 6]):
        b = oracle.average([grads[p] for p in perm])
        np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_cancellation_keeps_the_small_term():
    # {1, 2^-20, -1}: fp32 left-to-right would also keep it, but {2^-20, 1, -1} would
    # lose it; the exact sum keeps it in every order.
    one = np.array([0x3F80], dtype=np.uint16)
    small = np.array([(127 - 20) << 7], dtype=np.uint16)
    neg = np.array([0xBF80], dtype=np.uint16)
    for order in ([one, small, neg], [small, one, neg], [one, neg, small]):
        got = oracle.average(order)[0]
        assert got == np.float32(frac_to_f32(Fraction(2) ** -20 / 3))


# ---------------------------------------------------------------------------
# the optimizer half: Adam
# ---------------------------------------------------------------------------

def _torch_adam(theta0, grads_seq, lr, b1, b2, eps, wd=0.0, adamw=False):
    p = torch.nn.Parameter(torch.from_numpy(theta0.astype(np.float64)))
    cls = torch.optim.AdamW if adamw else torch.optim.Adam
    opt = cls([p], lr=float(np.float32(lr)), betas=(float(np.float32(b1)), float(np.float32(b2))),
              eps=float(np.float32(eps)), weight_decay=float(np.float32(wd)))
    out = []
    for g in grads_seq:
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
        out.append(p.detach().numpy().copy())
    return out


@pytest.mark.parametrize("hp", [
    dict(lr=1e-3, b1=0.9, b2=0.999, eps=1e-8),
    dict(lr=1e-2, b1=0.8, b2=0.95, eps=1e-3),     # eps comparable to |g|: placement matters
    dict(lr=3e-4, b1=0.5, b2=0.9, eps=0.0),
])
def test_adam_matches_torch_optim_adam_float64(hp):
    """torch.optim.Adam (textbook bias-corrected Adam, float64 states) agrees with
    the oracle within the effect of the oracle's fp32 state storage."""
    rng = np.random.default_rng(11)
    count, steps = 256, 4
    theta0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    gs = [(rng.standard_normal(count) * 1e-3 + 5e-4).astype(np.float32) for _ in range(steps)]
    ref = _torch_adam(theta0, gs, hp["lr"], hp["b1"], hp["b2"], hp["eps"])
    th, m, v = theta0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)
    for t, g in enumerate(gs, start=1):
        oracle.adam(g, th, m, v, lr=hp["lr"], beta1=hp["b1"], beta2=hp["b2"], eps=hp["eps"], step=t)
        tol = 8 * t * U * (np.abs(ref[t - 1]) + hp["lr"])
        np.testing.assert_array_less(np.abs(th - ref[t - 1]), tol + 1e-30)


def test_adamw_matches_torch_optim_adamw_float64():
    rng = np.random.default_rng(12)
    count, steps, lr, wd = 256, 3, 1e-2, 0.01
    theta0 = (rng.standard_normal(count) * 0.5).astype(np.float32)
    gs = [(rng.standard_normal(count) * 1e-3).astype(np.float32) for _ in range(steps)]
    ref = _torch_adam(theta0, gs, lr, 0.9, 0.999, 1e-8, wd=wd, adamw=True)
    th, m, v = theta0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)
    for t, g in enumerate(gs, start=1):
        oracle.adam(g, th, m, v, lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, step=t, weight_decay=wd)
        np.testing.assert_array_less(np.abs(th - ref[t - 1]),
                                     8 * t * U * (np.abs(ref[t - 1]) + lr))


def test_first_step_closed_form():
    """From m = v = 0: m_hat = g, v_hat = g^2, so delta = lr*g/(|g| + eps)."""
    rng = np.random.default_rng(13)
    count, lr, eps = 4096, 1e-3, 1e-8
    g = (rng.standard_normal(count) * 10.0 ** rng.integers(-9, 0, count)).astype(np.float32)
    th0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)
    out = oracle.adam(g, th, m, v, lr=lr, beta1=0.9, beta2=0.999, eps=eps, step=1)
    g64 = g.astype(np.float64)
    delta = np.float64(np.float32(lr)) * g64 / (np.abs(g64) + np.float64(np.float32(eps)))
    want = th0.astype(np.float64) - delta
    np.testing.assert_array_less(np.abs(th - want), U * np.abs(want) + 4 * U * np.abs(delta) + 1e-45)
    np.testing.assert_array_equal(m, (np.float64(1 - np.float64(np.float32(0.9))) * g64)
                                  .astype(np.float32))
    np.testing.assert_array_equal(out, oracle.f32_to_bf16(th))


def test_constant_gradient_closed_form():
    """Same g every step: m_hat_t = g and v_hat_t = g^2 for every t, so each step
    moves theta by lr*g/(|g|+eps)."""
    rng = np.random.default_rng(14)
    count, lr, eps, k = 2048, 1e-3, 1e-8, 6
    g = (rng.standard_normal(count) * 1e-3).astype(np.float32)
    th0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)
    for t in range(1, k + 1):
        oracle.adam(g, th, m, v, lr=lr, beta1=0.9, beta2=0.999, eps=eps, step=t)
    g64 = g.astype(np.float64)
    step = np.float64(np.float32(lr)) * g64 / (np.abs(g64) + np.float64(np.float32(eps)))
    want = th0.astype(np.float64) - k * step
    tol = k * (U * (np.abs(th0) + k * np.abs(step)) + 8 * U * np.abs(step))
    np.testing.assert_array_less(np.abs(th - want), tol)


def test_zero_gradient_leaves_master_unchanged():
    rng = np.random.default_rng(15)
    th0 = (rng.standard_normal(1000) * 0.02).astype(np.float32)
    th, m, v = th0.copy(), np.zeros(1000, np.float32), np.zeros(1000, np.float32)
    for t in (1, 2, 3):
        oracle.adam(np.zeros(1000, np.float32), th, m, v, lr=1e-3, beta1=0.9, beta2=0.999,
                    eps=1e-8, step=t)
    np.testing.assert_array_equal(th, th0)
    assert not m.any() and not v.any()


def test_zero_betas_reduce_to_normalised_step_every_step():
    """beta1 = beta2 = 0: m = g, v = g^2 and no bias correction, whatever the history."""
    rng = np.random.default_rng(16)
    count, lr, eps = 1024, 1e-2, 1e-8
    th = (rng.standard_normal(count) * 0.02).astype(np.float32)
    m = (rng.standard_normal(count)).astype(np.float32)
    v = np.abs(rng.standard_normal(count)).astype(np.float32)
    for t in (1, 5):
        g = (rng.standard_normal(count) * 1e-3).astype(np.float32)
        before = th.astype(np.float64)
        oracle.adam(g, th, m, v, lr=lr, beta1=0.0, beta2=0.0, eps=eps, step=t)
        np.testing.assert_array_equal(m, g)
        np.testing.assert_array_equal(v, (g.astype(np.float64) ** 2).astype(np.float32))
        g64 = g.astype(np.float64)
        want = before - np.float64(np.float32(lr)) * g64 / (np.abs(g64) + np.float64(np.float32(eps)))
        np.testing.assert_array_less(np.abs(th - want), U * np.abs(want) + 4 * U * lr)


def test_adam_is_invariant_to_gradient_scale_without_eps():
    """With eps = 0 Adam's step does not depend on a power-of-two rescaling of g."""
    rng = np.random.default_rng(17)
    count = 1024
    th0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    gs = [(rng.standard_normal(count) * 1e-3).astype(np.float32) for _ in range(3)]
    res = []
    for scale in (1.0, 2.0 ** 10, 2.0 ** -7):
        th, m, v = th0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)
        for t, g in enumerate(gs, start=1):
            oracle.adam((g * np.float32(scale)).astype(np.float32), th, m, v, lr=1e-3, beta1=0.9,
                        beta2=0.999, eps=0.0, step=t)
        res.append(th)
    np.testing.assert_array_equal(res[0], res[1])
    np.testing.assert_array_equal(res[0], res[2])


# ---------------------------------------------------------------------------
# composition: ZeRO shards, buckets
# ---------------------------------------------------------------------------

def test_zero_shards_concatenate_to_the_data_parallel_update():
    """ZeRO keeps data-parallel semantics: the N shard updates, concatenated,
    equal one update of the whole flattened vector."""
    rng = np.random.default_rng(18)
    n, numel = 4, 4 * 1000
    grads = [rand_bf16(rng, numel, -20, -5) for _ in range(n)]
    th0 = (rng.standard_normal(numel) * 0.02).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=1)
    th, m, v = th0.copy(), np.zeros(numel, np.float32), np.zeros(numel, np.float32)
    out_dp = oracle.reduce_adam_range(grads, 0, numel, th, m, v, **hp)
    s = numel // n
    parts = []
    for r in range(n):
        ths, ms, vs = th0[r * s:(r + 1) * s].copy(), np.zeros(s, np.float32), np.zeros(s, np.float32)
        parts.append((oracle.reduce_adam_shard(grads, numel, r, ths, ms, vs, **hp), ths))
    np.testing.assert_array_equal(np.concatenate([p[0] for p in parts]), out_dp)
    np.testing.assert_array_equal(np.concatenate([p[1] for p in parts]), th)


def test_shard_addressing_matches_printed_zero3_split():
    # 70B parameters, 64-way: 1/64 each ("Почему training 70B ...", §3-§4: 140/N GB of
    # fp16 parameters per GPU, ~2.2 GB at N=64, 17.5 GB at N=8)
    base, s = oracle.shard_range(70_000_000_000, 64, 5)
    assert s == 1_093_750_000 and base == 5 * s
    assert s * 2 == 2_187_500_000
    assert oracle.shard_range(70_000_000_000, 8, 0)[1] * 2 == 17_500_000_000
    with pytest.raises(ValueError):
        oracle.shard_range(10, 3, 0)
    with pytest.raises(ValueError):
        oracle.shard_range(12, 3, 3)


@pytest.mark.parametrize("shard,bucket", [(0, 5), (1, 1), (10, 3), (31_000_000, 25_000_000),
                                          (162_500_000, 50_000_000), (1_093_750_000, 4_000_000)])
def test_bucket_ranges_tile_the_shard(shard, bucket):
    rs = oracle.bucket_ranges(shard, bucket)
    assert sum(ln for _, ln in rs) == shard
    pos = 0
    for i, (off, ln) in enumerate(rs):
        assert off == pos and 0 < ln <= bucket
        if i < len(rs) - 1:
            assert ln == bucket
        pos += ln
    assert len(rs) == -(-shard // bucket)


def test_bucket_count_for_the_70b_shard():
    # 4M-element buckets ("M" decimal): 273 full buckets and a 1.75M-element tail
    rs = oracle.bucket_ranges(1_093_750_000, 4_000_000)
    assert len(rs) == 274 and rs[-1] == (273 * 4_000_000, 1_750_000)


# ---------------------------------------------------------------------------
# accounting against the printed figures
# ---------------------------------------------------------------------------

def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "state_accounting.txt"), encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split(None, 7)
            rows.append((float(parts[0]), int(parts[1]), int(parts[2]), int(parts[3]), parts[4],
                         float(parts[5]), parts[6], parts[7].strip()))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[7][:40])
def test_state_accounting_matches_printed_figures(row):
    psi, variant, n_dp, stage, comp, expected, rel, _cite = row
    comps = oracle.state_components(psi, variant, n_dp, stage)
    got = oracle.state_bytes(psi, variant, n_dp, stage) if comp == "total" else comps[comp]
    if rel == "eq":
        assert got == pytest.approx(expected, rel=1e-12)
    elif rel == "r1":   # printed to one decimal of a GB
        assert round(got / 1e8) == round(expected / 1e8), (got, expected)
    else:
        assert got > expected


def test_eight_a100s_hold_the_conservative_70b_replica():
    # "Почему training 70B ...", §2: at least 8 x A100 80 GB = 640 GB >= 560 GB
    total = oracle.state_bytes(70e9, 1, 1, 0)
    assert 8 * 80e9 >= total and 8 * 80e9 == 640e9


# ---------------------------------------------------------------------------
# gradient clipping (AdamW + global-norm clipping row)
# ---------------------------------------------------------------------------

def test_sqnorm_matches_exact_rational_sum_of_squares():
    rng = np.random.default_rng(21)
    n, count = 3, 300
    grads = [rand_bf16(rng, count, -12, 2) for _ in range(n)]
    g = oracle.average(grads)
    want = sum(Fraction(float(x)) ** 2 for x in g)
    got = oracle.grad_sqnorm(grads)
    assert abs(Fraction(got) - want) <= want * Fraction(1, 2 ** 45)
    # unscale by a power of two scales the squared norm exactly by its square
    assert oracle.grad_sqnorm(grads, unscale=0.25) == got / 16


def test_clipping_matches_torch_clip_grad_norm():
    """torch.nn.utils.clip_grad_norm_ (library, float64) on the averaged gradient of
    two 'shards' gives the same total norm and, after fp32 rounding, the same
    clipped gradient as the oracle."""
    rng = np.random.default_rng(22)
    n, numel = 4, 8000
    grads = [rand_bf16(rng, numel, -10, 0) for _ in range(n)]
    g = oracle.average(grads).astype(np.float64)
    for max_norm in (1e-3, 1.0, 1e6):
        t = torch.from_numpy(g.copy()).requires_grad_()
        t.grad = torch.from_numpy(g.copy())
        total = float(torch.nn.utils.clip_grad_norm_([t], max_norm))
        sq = oracle.grad_sqnorm(grads, 0, numel // 2) + oracle.grad_sqnorm(grads, numel // 2,
                                                                           numel // 2)
        assert np.sqrt(sq) == pytest.approx(total, rel=1e-14)
        c = oracle.grad_scale(sq, max_norm)
        ours = (g.astype(np.float32).astype(np.float64) * np.float64(c)).astype(np.float32)
        ref = t.grad.numpy()
        np.testing.assert_allclose(ours, ref, rtol=3 * U, atol=0)
        if max_norm >= 1e6:
            assert c == np.float32(1.0)


def test_clipped_adamw_step_equals_adamw_on_the_clipped_gradient():
    rng = np.random.default_rng(23)
    n, count = 2, 1000
    grads = [rand_bf16(rng, count, -12, 0) for _ in range(n)]
    th0 = (rng.standard_normal(count) * 0.02).astype(np.float32)
    c = oracle.grad_scale(oracle.grad_sqnorm(grads), 0.05)
    assert c < 1
    a = [th0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)]
    out_a = oracle.reduce_adamw_range(grads, 0, count, *a, lr=1e-3, beta1=0.9, beta2=0.999,
                                      eps=1e-8, step=1, weight_decay=0.01, gscale=float(c))
    g = (oracle.average(grads).astype(np.float64) * np.float64(c)).astype(np.float32)
    b = [th0.copy(), np.zeros(count, np.float32), np.zeros(count, np.float32)]
    out_b = oracle.adam(g, *b, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, step=1,
                        weight_decay=0.01)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    np.testing.assert_array_equal(out_a, out_b)


# ---------------------------------------------------------------------------
# fp16 gradients (fp16 + dynamic loss scaling row)
# ---------------------------------------------------------------------------

def test_f16_widening_matches_numpy_float16():
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(ours[fin], ref[fin])
    assert np.all(np.isnan(ours[np.isnan(ref)]))
    np.testing.assert_array_equal(ours[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_average_equals_exact_rational_average():
    rng = np.random.default_rng(31)
    n, count = 5, 400
    bits = [rng.integers(0, 0x7C00, count).astype(np.uint16) | (rng.integers(0, 2, count) << 15)
            .astype(np.uint16) for _ in range(n)]
    got = oracle.average([oracle.as_f16_bits(b) for b in bits])
    for j in range(count):
        s = sum(Fraction(float(np.uint16(b[j]).view(np.float16))) for b in bits)
        assert got[j] == np.float32(frac_to_f32(Fraction(frac_to_f32(s)) / n))


def test_loss_scaler_follows_the_worked_trajectory():
    rows = []
    with open(os.path.join(GOLDEN, "loss_scale_trajectory.txt"), encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            rows.append(line.split())
    cfg = rows[0]
    assert cfg[0] == "config"
    sc = oracle.LossScaler(float(cfg[1]), int(cfg[2]), int(cfg[3]), float(cfg[4]))
    for r in rows[1:]:
        sc.update(bool(int(r[0])))
        assert (sc.scale, sc.good_steps, sc.hysteresis_left, sc.step) == (
            float(r[1]), int(r[2]), int(r[3]), int(r[4])), r


def test_amp_step_on_power_of_two_scaled_fp16_grads_equals_the_unscaled_step():
    """Loss scaling by 2^k is exact on fp16 gradients that stay in range, so the
    unscaled step sees exactly the gradients of an unscaled run."""
    rng = np.random.default_rng(33)
    n, numel = 4, 4000
    raw = [(rng.standard_normal(numel) * 1e-3).astype(np.float16) for _ in range(n)]
    scaled = [oracle.as_f16_bits((r.astype(np.float32) * 1024).astype(np.float16).view(np.uint16))
              for r in raw]
    plain = [oracle.as_f16_bits(r.view(np.uint16)) for r in raw]
    # the scaled values are exactly 1024x the raw ones
    np.testing.assert_array_equal(oracle.f16_to_f64(scaled[0]), 1024 * raw[0].astype(np.float64))
    th0 = (rng.standard_normal(numel // n) * 0.02).astype(np.float32)
    a = [th0.copy(), np.zeros(th0.size, np.float32), np.zeros(th0.size, np.float32)]
    sc = oracle.LossScaler(1024.0, 1000, 2, 1.0)
    out_a, ovf = oracle.amp_step(scaled, 0, th0.size, *a, sc, lr=1e-3, beta1=0.9, beta2=0.999,
                                 eps=1e-8, weight_decay=0.01, max_grad_norm=1.0)
    assert not ovf and sc.step == 1
    b = [th0.copy(), np.zeros(th0.size, np.float32), np.zeros(th0.size, np.float32)]
    sc1 = oracle.LossScaler(1.0, 1000, 2, 1.0)
    out_b, _ = oracle.amp_step(plain, 0, th0.size, *b, sc1, lr=1e-3, beta1=0.9, beta2=0.999,
                               eps=1e-8, weight_decay=0.01, max_grad_norm=1.0)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    np.testing.assert_array_equal(out_a, out_b)


def test_amp_step_skips_on_overflow_and_leaves_the_states_alone():
    rng = np.random.default_rng(34)
    n, numel = 2, 1000
    g = [oracle.as_f16_bits((rng.standard_normal(numel) * 10).astype(np.float16).view(np.uint16))
         for _ in range(n)]
    g[1][777] = 0x7C00  # +Inf in one replica, in another rank's shard
    th0 = (rng.standard_normal(500) * 0.02).astype(np.float32)
    st = [th0.copy(), np.ones(500, np.float32), np.ones(500, np.float32)]
    sc = oracle.LossScaler(65536.0, 1000, 1, 1.0)
    out, ovf = oracle.amp_step(g, 0, 500, *st, sc, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    assert ovf and out is None and sc.step == 0 and sc.skipped == 1 and sc.scale == 32768.0
    np.testing.assert_array_equal(st[0], th0)
    assert np.all(st[1] == 1) and np.all(st[2] == 1)


def test_adam_matches_a_50_digit_decimal_evaluation():
    """The oracle's fp64 Adam against the same steps carried out in 50-digit
    decimal arithmetic (square root included), the stored states rounded to
    fp32 after every step as the method stores them: 16 elements x 3 steps,
    mixed signs and magnitudes, bit for bit."""
    import decimal
    from decimal import Decimal as D

    ctx = decimal.Context(prec=50)
    rng = np.random.default_rng(21)
    count, steps = 16, 3
    lr, b1, b2, eps = np.float32(1e-3), np.float32(0.9), np.float32(0.999), np.float32(1e-8)
    th = (rng.standard_normal(count) * 0.02).astype(np.float32)
    m = np.zeros(count, np.float32)
    v = np.zeros(count, np.float32)
    gs = [(rng.standard_normal(count) * 10.0 ** rng.integers(-6, -1, count)).astype(np.float32)
          for _ in range(steps)]
    dth, dm, dv = ([D(float(x)) for x in a] for a in (th, m, v))
    Dlr, Db1, Db2, Deps = (D(float(x)) for x in (lr, b1, b2, eps))
    f32 = lambda x: np.float32(float(x))          # noqa: E731 (decimal -> binary64 -> binary32)
    for t, g in enumerate(gs, start=1):
        oracle.adam(g, th, m, v, lr=float(lr), beta1=float(b1), beta2=float(b2), eps=float(eps),
                    step=t)
        bc1 = ctx.subtract(D(1), ctx.power(Db1, t))
        bc2 = ctx.subtract(D(1), ctx.power(Db2, t))
        for j in range(count):
            gj = D(float(g[j]))
            mn = ctx.add(ctx.multiply(Db1, dm[j]), ctx.multiply(ctx.subtract(D(1), Db1), gj))
            vn = ctx.add(ctx.multiply(Db2, dv[j]),
                         ctx.multiply(ctx.multiply(ctx.subtract(D(1), Db2), gj), gj))
            m32, v32 = f32(mn), f32(vn)
            mhat = ctx.divide(D(float(m32)), bc1)
            vhat = ctx.divide(D(float(v32)), bc2)
            delta = ctx.divide(ctx.multiply(Dlr, mhat), ctx.add(ctx.sqrt(vhat), Deps))
            th32 = f32(ctx.subtract(dth[j], delta))
            dm[j], dv[j], dth[j] = D(float(m32)), D(float(v32)), D(float(th32))
            assert m[j] == m32 and v[j] == v32 and th[j] == th32, (t, j)
