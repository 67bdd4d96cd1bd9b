"""The allocation-free squared-norm entry point (dpopt_grad_sqnorm_noalloc),
for callers that cannot allocate device scratch memory themselves.

Its answer must match the scratch-buffer entry point (dpopt_grad_sqnorm) on
the same inputs, call after call: the built-in partials array is shared by
every call and keeps the previous call's contents, so two calls in a row on
different inputs check that nothing stale leaks into the second answer.
Named to run last, so a failure here never hides the other tests' results."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import zero_mixed_precision_gb300 as dp
    return dp


def _grads(n, numel, step, dtype):
    """N flat gradient buffers of `numel` elements, seeded, on the device."""
    kind = 0 if dtype == torch.bfloat16 else 1
    out = []
    for r in range(n):
        buf = torch.empty(numel, dtype=dtype, device="cuda")
        synth.device_fill(buf.data_ptr(), kind, 0, numel, 77, synth.stream_id(1, r, step),
                          synth.Dist(r * 1e-5, 1e-3, outlier_p=0.01, outlier_scale=100.0))
        out.append(buf)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("n,S,dtype,unscale", [(4, 1_000_003, torch.bfloat16, 0.0),
                                               (8, 65_536 * 3, torch.float32, 0.25),
                                               (1, 7, torch.bfloat16, 0.0)])
def test_noalloc_matches_the_scratch_entry_point_twice_in_a_row(n, S, dtype, unscale):
    dp = _lib()
    gdt = dp.DPOPT_GRAD_BF16 if dtype == torch.bfloat16 else dp.DPOPT_GRAD_F32
    stream = torch.cuda.current_stream().cuda_stream
    rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)
    assert rc == 0
    scratch = torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")
    want = torch.zeros(1, dtype=torch.float64, device="cuda")
    got = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    for step in (1, 2):   # two calls in a row, different inputs
        grads = _grads(n, n * S, step, dtype)
        ptrs = [g.data_ptr() for g in grads]
        rank = n - 1
        assert dp.dpopt_grad_sqnorm(ptrs, gdt, n, n * S, rank, unscale, want.data_ptr(),
                                    scratch.data_ptr(), nbytes, stream) == 0
        assert dp.dpopt_grad_sqnorm_noalloc(ptrs, gdt, n, n * S, rank, unscale, got.data_ptr(),
                                            stream) == 0
        assert dp.dpopt_stream_status(stream) == 0
        w, g = float(want.item()), float(got.item())
        assert np.isfinite(g) and w > 0
        # the same kernels over the same fixed chunks in the same order: the
        # same bits, so a stale or misplaced partial cannot hide in a tolerance
        assert got.view(torch.int64).item() == want.view(torch.int64).item(), (g, w)
        # and the oracle's value: both sides sum S non-negative terms, the
        # oracle sequentially in fp64, so they agree within 4 S 2^-53 relative
        kind = 0 if dtype == torch.bfloat16 else 1
        host = [synth.host_fill(kind, rank * S, S, 77, synth.stream_id(1, r, step),
                                synth.Dist(r * 1e-5, 1e-3, outlier_p=0.01, outlier_scale=100.0))
                for r in range(n)]
        ref = oracle.grad_sqnorm(host, 0, S, unscale if unscale else 1.0)
        assert g == pytest.approx(ref, rel=4 * S * 2.0 ** -53)


def test_noalloc_rejects_shards_beyond_its_array():
    dp = _lib()
    fake = [0x10_0000_0000 + r * 0x1_0000_0000_00 for r in range(2)]
    too_big = 2 * ((1 << 31) + 1)            # one element past 2^31 per shard
    rc = dp.dpopt_grad_sqnorm_noalloc(fake, dp.DPOPT_GRAD_BF16, 2, too_big, 0, 0.0,
                                      0xF0_0000_0000, 0)
    assert rc == dp.DPOPT_ERR_UNSUPPORTED
    assert "2147483648" in dp.dpopt_last_error()


def test_noalloc_empty_shard_sets_up_and_writes_zero():
    """A call with an empty shard does only the device's set-up (the array's
    address) and writes 0, so callers can make it before a stream capture."""
    dp = _lib()
    out = torch.full((1,), float("nan"), dtype=torch.float64, device="cuda")
    g = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert dp.dpopt_grad_sqnorm_noalloc([g.data_ptr() or 0x10_0000_0000] * 2, dp.DPOPT_GRAD_BF16,
                                        2, 0, 0, 0.0, out.data_ptr(), stream) == 0
    assert dp.dpopt_stream_status(stream) == 0
    assert out.item() == 0.0
