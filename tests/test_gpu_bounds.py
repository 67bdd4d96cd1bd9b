"""The bounds-checked build (libdpopt_bounds.so) in place of a memory checker:
every kernel's derived indices are tested before the access.  The battery of
calls in tests/bounds_battery.py -- every kernel, ragged tails, unaligned
slices, batched launches, the bulk-copy kernel -- must run on it without a
single failed check and give bit for bit the release build's results; and the
deliberate failure of its self-test must reach dpopt_stream_status as
DPOPT_ERR_BOUNDS exactly once."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_checked_build_is_silent_and_bitwise_equal(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import bounds_battery
    import zero_mixed_precision_gb300 as dp

    path = tmp_path / "bounds.npz"
    env = dict(os.environ, DPOPT_LIB_VARIANT="bounds")
    pr = subprocess.run([sys.executable, "-m", "tests.bounds_battery", str(path)], cwd=ROOT,
                        env=env, capture_output=True, text=True, timeout=600)
    assert pr.returncode == 0, pr.stdout + pr.stderr
    got = np.load(path)
    assert str(got["__version__"]).endswith("+bounds")
    # every call's status: no index check failed anywhere
    bad = [(n, int(s)) for n, s in zip(got["__names__"], got["__status__"]) if s != 0]
    assert not bad, bad
    # the self-test: enqueued, reported as DPOPT_ERR_BOUNDS once, then cleared
    assert got["__selftest__"].tolist() == [dp.DPOPT_OK, dp.DPOPT_ERR_BOUNDS, dp.DPOPT_OK]

    assert not dp.dpopt_version().endswith("+bounds")
    want, status = bounds_battery.run()
    assert all(s == 0 for _, s in status), status
    keys = sorted(k for k in got.files if not k.startswith("__"))
    assert keys == sorted(want)
    for k in keys:
        a, b = want[k], got[k]
        assert a.dtype == b.dtype and a.shape == b.shape, k
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), k
