"""Compile the CUDA library in-tree for sm_103a (the only target).

The library is several translation units compiled in parallel and linked
into one shared object: the C ABI (dpopt.cu), the bulk-copy kernel (tma.cu)
and the kernels of each gradient type (launch_gk.cu, once per type)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
LIB_PATH = os.path.join(LIB_DIR, "libdpopt.so")

# (object name, source, extra flags)
UNITS = [
    ("dpopt", "dpopt.cu", []),
    ("tma", "tma.cu", []),
    ("step_bf16", "launch_gk.cu", ["-DDPOPT_GK=0"]),
    ("step_f32", "launch_gk.cu", ["-DDPOPT_GK=1"]),
    ("step_f16", "launch_gk.cu", ["-DDPOPT_GK=2"]),
]
SOURCES = sorted({os.path.join(CSRC, src) for _, src, _ in UNITS})
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                     if f.endswith((".cuh", ".h"))] + [os.path.join(INCLUDE, "dpopt.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH,
    "-O3", "-lineinfo", "-std=c++17",
    "-prec-div=true", "-prec-sqrt=true", "-fmad=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
]


def object_path(name: str) -> str:
    return os.path.join(OBJ_DIR, name + ".o")


def compile_command(name: str, src: str, extra: list[str]) -> list[str]:
    return ["nvcc", *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
            os.path.join(CSRC, src), "-o", object_path(name)]


def link_command() -> list[str]:
    return ["nvcc", *ARCH, "-shared", *[object_path(n) for n, _, _ in UNITS], "-o", LIB_PATH]


def stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False) -> str:
    os.makedirs(OBJ_DIR, exist_ok=True)
    if force or stale():
        with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
            procs = list(ex.map(lambda u: subprocess.run(compile_command(*u), capture_output=True,
                                                         text=True), UNITS))
        for (name, _, _), pr in zip(UNITS, procs):
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed for {name}:\n{pr.stdout}{pr.stderr}")
        subprocess.run(link_command(), check=True)
    return LIB_PATH
