"""CPU oracle for the fused ZeRO reduce + mixed-precision Adam step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
baseline leg of the benchmark may import this package.  The product path
(the CUDA library and its Python binding) never imports, links or runs it,
and it shares no code with that path: the arithmetic lives in ``oracle.c``
(plain fp64 C) and in the pure-Python helpers below.

Pins: every function here is checked in ``tests/test_oracle_pins.py``
against something other than itself (printed figures of the pages, closed
forms, brute force with exact rationals, and library routines).  No
function is "parity unpinned".

Sources: see the header of ``oracle.c``; the accounting helpers restate
"Глава 4.4 -- Распределённое обучение" §2 and §6, and
"Почему training 70B модели требует optimizer sharding (ZeRO-3)?" §2-§4.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

GRAD_BF16 = 0
GRAD_F32 = 1
GRAD_F16 = 2


def build_command() -> list[str]:
    """The compiler line for the oracle (plain C, IEEE arithmetic, OpenMP)."""
    return ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", "-fopenmp", _SRC, "-o", _LIB_PATH, "-lm"]


def build() -> str:
    subprocess.run(build_command(), check=True)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        L = ctypes.CDLL(_LIB_PATH)
        P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_f32_to_bf16_rne.argtypes = [F]
        L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
        L.orc_reduce_adam_range.argtypes = [P, I, I, I64, I64, P, P, P, P, F, F, F, F, F, I64, I]
        L.orc_reduce_adam_range.restype = I
        L.orc_reduce_adam_shard.argtypes = [P, I, I, I64, I, P, P, P, P, F, F, F, F, F, I64, I]
        L.orc_reduce_adam_shard.restype = I
        L.orc_reduce_adam_gathered.argtypes = [P, I, I, I64, P, P, P, P, F, F, F, F, F, I64]
        L.orc_reduce_adam_gathered.restype = I
        L.orc_average.argtypes = [P, I, I, I64, P]
        L.orc_average.restype = I
        L.orc_adam.argtypes = [P, I64, P, P, P, P, F, F, F, F, F, I64]
        L.orc_adam.restype = I
        L.orc_f32_to_bf16_array.argtypes = [P, I64, P]
        L.orc_f32_to_bf16_array.restype = None
        L.orc_threads_available.argtypes = []
        L.orc_threads_available.restype = I
        L.orc_f16_to_f64_array.argtypes = [P, I64, P]
        L.orc_f16_to_f64_array.restype = None
        L.orc_grad_sqnorm.argtypes = [P, I, I, I64, I64, F]
        L.orc_grad_sqnorm.restype = ctypes.c_double
        L.orc_grad_scale.argtypes = [ctypes.c_double, F, F]
        L.orc_grad_scale.restype = F
        L.orc_reduce_adamw_range.argtypes = [P, I, I, I64, I64, P, P, P, P, F, F, F, F, F, F, I64]
        L.orc_reduce_adamw_range.restype = I
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# array marshalling
# ---------------------------------------------------------------------------

class F16Bits(np.ndarray):
    """uint16 array holding binary16 bit patterns (plain uint16 arrays are read
    as bf16)."""


def as_f16_bits(a: np.ndarray) -> "F16Bits":
    return np.ascontiguousarray(a, dtype=np.uint16).view(F16Bits)


def _dtype_code(arr: np.ndarray) -> int:
    if isinstance(arr, F16Bits):
        return GRAD_F16
    if arr.dtype == np.uint16:
        return GRAD_BF16
    if arr.dtype == np.float32:
        return GRAD_F32
    raise TypeError(f"gradients must be bf16/fp16 bit patterns (uint16) or float32, got {arr.dtype}")


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _ptr_table(grads: Sequence[np.ndarray]):
    table = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    return table


def _check_rc(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid argument")


# ---------------------------------------------------------------------------
# the method
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of binary16 bit patterns to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().orc_f16_to_f64_array(_ptr(b), b.size, _ptr(out))
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even bf16 bit patterns of a float32 array."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def _contig(g: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(g)
    return c.view(F16Bits) if isinstance(g, F16Bits) else c


def average(grads: Sequence[np.ndarray]) -> np.ndarray:
    """Fixed-order (ascending replica) average of N equal-length gradient arrays."""
    grads = [_contig(g) for g in grads]
    n = len(grads)
    count = grads[0].size
    code = _dtype_code(grads[0])
    for g in grads:
        assert g.size == count and _dtype_code(g) == code
    out = np.empty(count, dtype=np.float32)
    _check_rc(lib().orc_average(_ptr_table(grads), code, n, count, _ptr(out)), "average")
    return out


def adam(g: np.ndarray, master: np.ndarray, m: np.ndarray, v: np.ndarray, *, lr: float,
         beta1: float, beta2: float, eps: float, step: int, weight_decay: float = 0.0):
    """One Adam step from an fp32 averaged gradient; updates master/m/v in place,
    returns the bf16 working copy (uint16 bit patterns)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == g.size
    out = np.empty(g.size, dtype=np.uint16)
    _check_rc(lib().orc_adam(_ptr(g), g.size, _ptr(master), _ptr(m), _ptr(v), _ptr(out),
                             lr, beta1, beta2, eps, weight_decay, step), "adam")
    return out


def reduce_adam_range(grads: Sequence[np.ndarray], offset: int, count: int, master: np.ndarray,
                      m: np.ndarray, v: np.ndarray, *, lr: float, beta1: float, beta2: float,
                      eps: float, step: int, weight_decay: float = 0.0, nthreads: int = 1):
    """Average N flattened replica buffers over [offset, offset+count) and apply
    one Adam step to the count-element states (in place).  Returns the bf16
    working copy."""
    grads = [_contig(g) for g in grads]
    code = _dtype_code(grads[0])
    for g in grads:
        assert _dtype_code(g) == code and g.size >= offset + count
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == count
    out = np.empty(count, dtype=np.uint16)
    _check_rc(lib().orc_reduce_adam_range(_ptr_table(grads), code, len(grads), offset, count,
                                          _ptr(master), _ptr(m), _ptr(v), _ptr(out), lr, beta1,
                                          beta2, eps, weight_decay, step, nthreads),
              "reduce_adam_range")
    return out


def reduce_adam_shard(grads: Sequence[np.ndarray], numel: int, shard_rank: int, master, m, v, *,
                      lr: float, beta1: float, beta2: float, eps: float, step: int,
                      weight_decay: float = 0.0, nthreads: int = 1):
    """ZeRO shard form: rank shard_rank of N = len(grads) updates [r*S, (r+1)*S)."""
    n = len(grads)
    if n < 1 or numel % n != 0 or not 0 <= shard_rank < n:
        raise ValueError("oracle reduce_adam_shard: invalid argument")
    s = numel // n
    return reduce_adam_range(grads, shard_rank * s, s, master, m, v, lr=lr, beta1=beta1,
                             beta2=beta2, eps=eps, step=step, weight_decay=weight_decay,
                             nthreads=nthreads)


def grad_sqnorm(grads: Sequence[np.ndarray], offset: int = 0, count: int | None = None,
                unscale: float = 1.0) -> float:
    """sum of (g_i * unscale)^2 over [offset, offset+count) of the averaged gradient."""
    grads = [_contig(g) for g in grads]
    code = _dtype_code(grads[0])
    count = grads[0].size - offset if count is None else count
    return float(lib().orc_grad_sqnorm(_ptr_table(grads), code, len(grads), offset, count,
                                       unscale))


def grad_scale(sqnorm: float, max_norm: float, unscale: float = 1.0) -> np.float32:
    """fp32 multiplier unscale * min(1, max_norm / (sqrt(sqnorm) + 1e-6))."""
    return np.float32(lib().orc_grad_scale(sqnorm, max_norm, unscale))


def reduce_adamw_range(grads: Sequence[np.ndarray], offset: int, count: int, master, m, v, *,
                       lr: float, beta1: float, beta2: float, eps: float, step: int,
                       weight_decay: float = 0.0, gscale: float = 1.0):
    """One AdamW step with the averaged gradient multiplied by gscale first."""
    grads = [_contig(g) for g in grads]
    code = _dtype_code(grads[0])
    for a in (master, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == count
    out = np.empty(count, dtype=np.uint16)
    _check_rc(lib().orc_reduce_adamw_range(_ptr_table(grads), code, len(grads), offset, count,
                                           _ptr(master), _ptr(m), _ptr(v), _ptr(out), lr, beta1,
                                           beta2, eps, weight_decay, gscale, step),
              "reduce_adamw_range")
    return out


def threads_available() -> int:
    return int(lib().orc_threads_available())


# ---------------------------------------------------------------------------
# addressing: the shard and its fusion buckets
# ---------------------------------------------------------------------------

def shard_range(numel: int, n_replicas: int, shard_rank: int) -> tuple[int, int]:
    """(base, S): rank r of N keeps the contiguous 1/N slice [r*S, (r+1)*S)
    ("Почему training 70B ...", §3: each GPU keeps only its part, 1/N of the
    total; §5: reduce-scatter keeps only its own shard)."""
    if n_replicas < 1 or numel < 0 or numel % n_replicas or not 0 <= shard_rank < n_replicas:
        raise ValueError("shard_range: invalid argument")
    s = numel // n_replicas
    return shard_rank * s, s


def bucket_ranges(shard_elems: int, bucket_elems: int) -> list[tuple[int, int]]:
    """Cut a shard into fusion buckets of bucket_elems elements from its start,
    the last one ragged (DeepSpeed's reduce_bucket_size over contiguous
    gradients, in the config of "Почему training 70B ...", §8)."""
    if shard_elems < 0 or bucket_elems < 1:
        raise ValueError("bucket_ranges: invalid argument")
    out = []
    off = 0
    while off < shard_elems:
        ln = min(bucket_elems, shard_elems - off)
        out.append((off, ln))
        off += ln
    return out


# ---------------------------------------------------------------------------
# model-state accounting
# ---------------------------------------------------------------------------

# bytes per parameter: (16-bit params, 16-bit grads, optimizer states)
_VARIANTS = {
    # mixed-precision Adam: fp16/bf16 param 2 + grad 2 + fp32 master 4 + m 4 + v 4
    # ("Глава 4.4" §2: 16*Psi bytes; DP page appendix: 16 bytes per parameter)
    0: (2, 2, 12),
    # the ZeRO-3 answer's "conservative" 70B figure: 140 GB params + 140 GB grads
    # + 280 GB optimizer = 560 GB, i.e. 2 + 2 + 4 bytes per parameter as printed
    # ("Почему training 70B ...", §2; its 280 GB is 4 B/param although the same
    # paragraph prices two fp32 moments at 8 B -- the printed total is kept)
    1: (2, 2, 4),
}


def state_components(psi: int | float, variant: int, n_dp: int,
                     zero_stage: int) -> dict[str, float]:
    """Model-state bytes held by ONE data-parallel device, by component.

    Stage 0 (plain DP) keeps everything; stage 1 shards the optimizer states,
    stage 2 also the gradients ("ZeRO-2 ... leaves a full copy of the
    parameters on each GPU", ZeRO-3 answer §4), stage 3 shards all three
    ("Глава 4.4" §6: about 16*Psi/N_dp at the most aggressive stage)."""
    if variant not in _VARIANTS or n_dp < 1 or zero_stage not in (0, 1, 2, 3) or psi < 0:
        raise ValueError("state_components: invalid argument")
    p, g, o = _VARIANTS[variant]
    psi = float(psi)
    shard_p = zero_stage >= 3
    shard_g = zero_stage >= 2
    shard_o = zero_stage >= 1
    return {
        "params": psi * p / (n_dp if shard_p else 1),
        "grads": psi * g / (n_dp if shard_g else 1),
        "optimizer": psi * o / (n_dp if shard_o else 1),
    }


def state_bytes(psi: int | float, variant: int, n_dp: int, zero_stage: int) -> float:
    """Total model-state bytes held by one device (sum of state_components)."""
    c = state_components(psi, variant, n_dp, zero_stage)
    return c["params"] + c["grads"] + c["optimizer"]


# ---------------------------------------------------------------------------
# dynamic loss scaling (the fp16 block of the ZeRO-3 answer's DeepSpeed config:
# loss_scale 0 = dynamic, initial_scale_power 16, loss_scale_window 1000,
# hysteresis 2, min_loss_scale 1).  The pages give only the keys; the reading:
#   - a step overflows when any averaged gradient element of any rank is not
#     finite (its global squared norm is then not finite);
#   - an overflowing step is skipped: no state changes, the step count stays;
#     the run of clean steps restarts; every `hysteresis`-th overflow since the
#     scale last changed halves the scale (never below min_scale);
#   - a clean step is applied to g / scale; after `window` clean steps in a row
#     the scale doubles.
# ---------------------------------------------------------------------------

class LossScaler:
    def __init__(self, init_scale: float = 2.0 ** 16, window: int = 1000, hysteresis: int = 2,
                 min_scale: float = 1.0):
        self.scale = float(init_scale)
        self.window = int(window)
        self.hysteresis = int(hysteresis)
        self.min_scale = float(min_scale)
        self.good_steps = 0
        self.hysteresis_left = int(hysteresis)
        self.step = 0          # optimizer steps taken
        self.skipped = 0

    def update(self, overflow: bool) -> None:
        if overflow:
            self.skipped += 1
            self.good_steps = 0
            self.hysteresis_left -= 1
            if self.hysteresis_left <= 0:
                self.scale = max(self.scale / 2.0, self.min_scale)
                self.hysteresis_left = self.hysteresis
        else:
            self.step += 1
            self.good_steps += 1
            if self.good_steps >= self.window:
                self.scale *= 2.0
                self.good_steps = 0
                self.hysteresis_left = self.hysteresis


def amp_step(all_grads, shard_offset: int, shard_len: int, master, m, v, scaler: LossScaler, *,
             lr: float, beta1: float, beta2: float, eps: float, weight_decay: float = 0.0,
             max_grad_norm: float = 0.0):
    """One mixed-precision step with dynamic loss scaling on one rank's shard.

    all_grads: the N replica buffers (scaled gradients, e.g. fp16) over the whole
    model, so the global norm and the overflow decision see every rank.  Updates
    master/m/v in place unless the step overflows; updates the scaler.  Returns
    (bf16 working copy or None if skipped, overflow)."""
    unscale = 1.0 / scaler.scale
    sq = grad_sqnorm(all_grads, 0, all_grads[0].size, unscale)
    overflow = not np.isfinite(sq)
    out = None
    if not overflow:
        gscale = grad_scale(sq, max_grad_norm, unscale)
        out = reduce_adamw_range(all_grads, shard_offset, shard_len, master, m, v, lr=lr,
                                 beta1=beta1, beta2=beta2, eps=eps, step=scaler.step + 1,
                                 weight_decay=weight_decay, gscale=float(gscale))
    scaler.update(overflow)
    return out, overflow
