"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds no arithmetic of the method.  It draws gradients and
optimizer states from a counter-based generator (definition in ``synth.c``)
that exists twice: a host version (``synth.c``, used for the oracle's inputs
and for any sampled element) and a device version (``synth_dev.cu``, used to
fill device memory for workloads too large to pass through the host).  The two
agree bit-for-bit; a GPU test checks it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .workloads import (  # noqa: F401  (re-export)
    Dist, Workload, WORKLOADS, SWEEP_SIZES, SWEEP_REPLICAS, STREAM_GRAD, STREAM_MASTER,
    STREAM_M, STREAM_V, stream_id, sweep_cell,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_SRC = os.path.join(_HERE, "synth.c")
_HOST_LIB = os.path.join(_HERE, "libsynth.so")
_DEV_SRC = os.path.join(_HERE, "synth_dev.cu")
_DEV_LIB = os.path.join(_HERE, "libsynth_dev.so")

KIND_BF16 = 0
KIND_F32 = 1
KIND_F16 = 2


def host_build_command() -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", _HOST_SRC, "-o", _HOST_LIB]


def device_build_command() -> list[str]:
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "-fmad=false", _DEV_SRC, "-o", _DEV_LIB]


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


_host = None
_dev = None


def _host_lib() -> ctypes.CDLL:
    global _host
    if _host is None:
        if _stale(_HOST_LIB, _HOST_SRC):
            subprocess.run(host_build_command(), check=True)
        L = ctypes.CDLL(_HOST_LIB)
        P, I, I64, U64, D = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                             ctypes.c_double)
        L.syn_fill.argtypes = [P, I, I64, I64, U64, U64, D, D, D, D, I]
        L.syn_fill.restype = None
        L.syn_gather.argtypes = [P, I, P, I64, U64, U64, D, D, D, D, I]
        L.syn_gather.restype = None
        L.syn_key.argtypes = [U64, U64]
        L.syn_key.restype = U64
        _host = L
    return _host


def _dev_lib() -> ctypes.CDLL:
    global _dev
    if _dev is None:
        if _stale(_DEV_LIB, _DEV_SRC):
            subprocess.run(device_build_command(), check=True)
        L = ctypes.CDLL(_DEV_LIB)
        P, I, I64, U64, D = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                             ctypes.c_double)
        L.syn_fill_device.argtypes = [P, I, I64, I64, U64, U64, D, D, D, D, I, P]
        L.syn_fill_device.restype = I
        _dev = L
    return _dev


def build_host() -> None:
    _host_lib()


def _dist_args(d: Dist):
    return (float(d.mu), float(d.sigma), float(d.outlier_p), float(d.outlier_scale),
            int(d.absval))


def host_fill(kind: int, start: int, count: int, seed: int, stream: int, dist: Dist) -> np.ndarray:
    """Elements start .. start+count-1 of one stream, as uint16 bf16 bits
    (kind 0), float32 (kind 1) or uint16 fp16 bits (kind 2)."""
    out = np.empty(count, dtype=np.float32 if kind == KIND_F32 else np.uint16)
    if count:
        _host_lib().syn_fill(out.ctypes.data, kind, start, count, seed, stream, *_dist_args(dist))
    return out


def host_gather(kind: int, idx: np.ndarray, seed: int, stream: int, dist: Dist) -> np.ndarray:
    """Elements idx[k] of one stream."""
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.size, dtype=np.float32 if kind == KIND_F32 else np.uint16)
    if idx.size:
        _host_lib().syn_gather(out.ctypes.data, kind, idx.ctypes.data, idx.size, seed, stream,
                               *_dist_args(dist))
    return out


def device_fill(ptr: int, kind: int, start: int, count: int, seed: int, stream: int, dist: Dist,
                cuda_stream: int = 0) -> None:
    """Fill device memory at ``ptr`` with the same elements host_fill gives."""
    rc = _dev_lib().syn_fill_device(ptr, kind, start, count, seed, stream, *_dist_args(dist),
                                    cuda_stream)
    if rc != 0:
        raise RuntimeError(f"syn_fill_device failed with cudaError {rc}")
