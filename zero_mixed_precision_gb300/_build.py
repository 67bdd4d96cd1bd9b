"""Compile the CUDA library in-tree for sm_103a (the only target)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libdpopt.so")
SOURCES = [os.path.join(CSRC, "dpopt.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(INCLUDE, "dpopt.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-prec-div=true", "-prec-sqrt=true", "-fmad=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
    "-shared",
]


def command() -> list[str]:
    return ["nvcc", *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, *SOURCES, "-o", LIB_PATH]


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False) -> str:
    os.makedirs(LIB_DIR, exist_ok=True)
    if force or stale():
        subprocess.run(command(), check=True)
    return LIB_PATH
