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

# Library variants: the release build, and the bounds-checked build whose
# kernels test every derived index before the access (-DDPOPT_DEBUG_BOUNDS).
VARIANTS = {
    "release": ("libdpopt.so", "obj", []),
    "bounds": ("libdpopt_bounds.so", "obj_bounds", ["-DDPOPT_DEBUG_BOUNDS"]),
}


def lib_path(variant: str = "release") -> str:
    return os.path.join(LIB_DIR, VARIANTS[variant][0])

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
    # host arithmetic (the step's fp64 scalars) rounds every operation on its
    # own on x86 and Arm alike: no fused multiply-add contraction
    "-Xcompiler", "-ffp-contract=off",
]


def object_path(name: str, variant: str = "release") -> str:
    return os.path.join(LIB_DIR, VARIANTS[variant][1], name + ".o")


def compile_command(name: str, src: str, extra: list[str], variant: str = "release") -> list[str]:
    os.makedirs(os.path.join(LIB_DIR, VARIANTS[variant][1]), exist_ok=True)
    return ["nvcc", *NVCC_FLAGS, *VARIANTS[variant][2], *extra, "-I", INCLUDE, "-I", CSRC, "-c",
            os.path.join(CSRC, src), "-o", object_path(name, variant)]


def link_command(variant: str = "release") -> list[str]:
    return ["nvcc", *ARCH, "-shared", *[object_path(n, variant) for n, _, _ in UNITS], "-o",
            lib_path(variant)]


def stale(variant: str = "release") -> bool:
    path = lib_path(variant)
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, variant: str = "release") -> str:
    if force or stale(variant):
        with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
            procs = list(ex.map(lambda u: subprocess.run(compile_command(*u, variant=variant),
                                                         capture_output=True, text=True), UNITS))
        for (name, _, _), pr in zip(UNITS, procs):
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed for {name}:\n{pr.stdout}{pr.stderr}")
        subprocess.run(link_command(variant), check=True)
    return lib_path(variant)
