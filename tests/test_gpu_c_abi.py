"""The C ABI from a plain C program (tests/c/abi_step.c): no Python or PyTorch
between the caller and the library -- cudaMalloc'd buffers, a cudaStream_t,
two steps of dpopt_reduce_adam, dpopt_stream_status, and the results checked
against the oracle's C entry point."""
from __future__ import annotations

import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_program_steps_through_the_abi(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = os.path.join(ROOT, "zero_mixed_precision_gb300", "lib")
    orc = os.path.join(ROOT, "oracle")
    exe = tmp_path / "abi_step"
    subprocess.run(["nvcc", "-x", "c", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c", "abi_step.c"), "-o", str(exe), "-L", lib,
                    "-ldpopt", "-L", orc, "-loracle", "-Xlinker", f"-rpath,{lib}:{orc}", "-lm"],
                   check=True)
    pr = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert pr.returncode == 0, pr.stdout + pr.stderr
    assert pr.stdout.startswith("ok:"), pr.stdout
    assert "bucket table bitwise equal" in pr.stdout
    assert "graph replays bitwise equal" in pr.stdout
