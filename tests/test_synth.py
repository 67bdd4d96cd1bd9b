"""Host side of the seeded input generator (no GPU)."""
import numpy as np

import synth


def test_gather_equals_fill_at_the_same_indices():
    d = synth.Dist(0.0, 1e-3, outlier_p=0.01, outlier_scale=100.0)
    s = synth.stream_id(synth.STREAM_GRAD, 3, 7)
    full = synth.host_fill(0, 1000, 50_000, 1, s, d)
    idx = np.array([1000, 1001, 25_000, 50_999, 33_333], dtype=np.int64)
    np.testing.assert_array_equal(synth.host_gather(0, idx, 1, s, d), full[idx - 1000])


def test_streams_and_seeds_are_independent_and_reproducible():
    d = synth.Dist(0.0, 1.0)
    a = synth.host_fill(1, 0, 10_000, 0, synth.stream_id(1, 0, 1), d)
    b = synth.host_fill(1, 0, 10_000, 0, synth.stream_id(1, 1, 1), d)
    c = synth.host_fill(1, 0, 10_000, 1, synth.stream_id(1, 0, 1), d)
    a2 = synth.host_fill(1, 0, 10_000, 0, synth.stream_id(1, 0, 1), d)
    np.testing.assert_array_equal(a, a2)
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.05 and abs(np.corrcoef(a, c)[0, 1]) < 0.05


def test_distribution_moments_and_outlier_rate():
    x = synth.host_fill(1, 0, 400_000, 5, 9, synth.Dist(0.25, 2.0)).astype(np.float64)
    assert abs(x.mean() - 0.25) < 0.02 and abs(x.std() - 2.0) < 0.02
    d = synth.Dist(0.0, 1.0, outlier_p=0.01, outlier_scale=100.0)
    y = synth.host_fill(1, 0, 400_000, 5, 9, d).astype(np.float64)
    rate = np.mean(np.abs(y) > 6.0)   # Irwin-Hall(12) never exceeds 6 sigma
    assert 0.008 < rate < 0.012
    v = synth.host_fill(1, 0, 10_000, 5, 9, synth.Dist(0.0, 1e-8, absval=True))
    assert np.all(v >= 0)


def test_bf16_kind_is_the_rounded_fp32_kind():
    d = synth.Dist(0.0, 1e-3)
    f = synth.host_fill(1, 0, 20_000, 2, 3, d)
    h = synth.host_fill(0, 0, 20_000, 2, 3, d)
    import torch
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(h, ref)


def test_fp16_kind_is_the_rounded_fp32_kind():
    """The host's binary16 rounding against numpy's (library), over the whole
    binary16 range: normal, subnormal, underflow to zero, overflow to Inf."""
    for sigma in (1e-3, 1.0, 3e3, 1e5, 1e-6, 1e-8):
        d = synth.Dist(0.0, sigma, outlier_p=0.05, outlier_scale=100.0)
        f = synth.host_fill(1, 0, 50_000, 3, 4, d)
        h = synth.host_fill(2, 0, 50_000, 3, 4, d)
        ref = f.astype(np.float16).view(np.uint16)
        np.testing.assert_array_equal(h, ref)
