"""Thin ctypes binding of libdpopt.so (include/dpopt.h).

Argument marshalling only: every step of the reduce + Adam path runs in the
CUDA kernels of the library.  The ``dpopt_*`` functions take the C ABI's
arguments (device pointers as ints, a stream handle as an int); the
lower-case wrappers below take torch tensors and pass their data pointers.
If the library is missing this module raises at import: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

from . import _build

DPOPT_OK = 0
DPOPT_ERR_INVALID_ARG = 1
DPOPT_ERR_UNSUPPORTED = 2
DPOPT_ERR_CUDA = 3
DPOPT_ERR_TIMEOUT = 4
DPOPT_ERR_BOUNDS = 5
DPOPT_GRAD_BF16 = 0
DPOPT_GRAD_F32 = 1
DPOPT_GRAD_F16 = 2
DPOPT_MAX_REPLICAS = 64
DPOPT_KERNEL_AUTO = 0
DPOPT_KERNEL_DIRECT = 1
DPOPT_KERNEL_BULK = 2
DPOPT_GATHER_AUTO = 0
DPOPT_GATHER_FUSED = 1
DPOPT_GATHER_SEPARATE = 2

# DPOPT_LIB_VARIANT=bounds loads the bounds-checked build of the same sources
# (every kernel tests its derived indices; failures are reported as
# DPOPT_ERR_BOUNDS by dpopt_stream_status); unset or "release": the release build.
LIB_VARIANT = os.environ.get("DPOPT_LIB_VARIANT", "release")
if LIB_VARIANT not in _build.VARIANTS:
    raise ImportError(f"DPOPT_LIB_VARIANT={LIB_VARIANT!r}: expected one of {sorted(_build.VARIANTS)}")
LIB_PATH = _build.lib_path(LIB_VARIANT)

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_PP = ctypes.POINTER(ctypes.c_void_p)
_PI64 = ctypes.POINTER(ctypes.c_int64)


class StepOptions(ctypes.Structure):
    """dpopt_step_options (include/dpopt.h)."""
    _fields_ = [("weight_decay", ctypes.c_float), ("max_grad_norm", ctypes.c_float),
                ("grad_sqnorm", ctypes.c_void_p), ("grad_unscale", ctypes.c_float)]


_POPT = ctypes.POINTER(StepOptions)


class LossScaleState(ctypes.Structure):
    """dpopt_loss_scale_state (device-resident; this is its host-side layout)."""
    _fields_ = [("scale", ctypes.c_float), ("good_steps", ctypes.c_int32),
                ("hysteresis_left", ctypes.c_int32), ("last_overflow", ctypes.c_int32),
                ("step", ctypes.c_int64), ("skipped", ctypes.c_int64)]


class LossScaleConfig(ctypes.Structure):
    """dpopt_loss_scale_config."""
    _fields_ = [("init_scale", ctypes.c_float), ("window", ctypes.c_int32),
                ("hysteresis", ctypes.c_int32), ("min_scale", ctypes.c_float)]


_PCFG = ctypes.POINTER(LossScaleConfig)

_SIGS = {
    "dpopt_reduce_adam": ([_PP, _I, _I64, _I, _I64, _P, _P, _P, _P, _F, _F, _F, _F, _I64, _P], _I),
    "dpopt_reduce_adam_ex": ([_PP, _I, _I, _I64, _I, _I64, _P, _P, _P, _P, _F, _F, _F, _F, _I64,
                              _P], _I),
    "dpopt_bucket_count": ([_I64, _I64, _PI64], _I),
    "dpopt_bucket_range": ([_I64, _I64, _I64, _PI64, _PI64], _I),
    "dpopt_reduce_adam_bucket": ([_PP, _I, _I, _I64, _I64, _P, _P, _P, _P, _F, _F, _F, _F, _I64,
                                  _P], _I),
    "dpopt_reduce_adam_buckets": ([_PP, _I, _I, _PI64, _PI64, _I64, _P, _P, _P, _P, _F, _F, _F, _F,
                                   _I64, _P], _I),
    "dpopt_bucket_table_bytes": ([_I, _I64, _PI64], _I),
    "dpopt_reduce_adam_buckets_table": ([_PP, _I, _I, _PI64, _PI64, _I64, _P, _P, _P, _P, _F, _F,
                                         _F, _F, _I64, _POPT, _P, _I64, _P], _I),
    "dpopt_stream_status": ([_P], _I),
    "dpopt_status_string": ([_I], ctypes.c_char_p),
    "dpopt_last_error": ([], ctypes.c_char_p),
    "dpopt_state_bytes": ([_I64, _I, _I, _I, ctypes.POINTER(ctypes.c_double)], _I),
    "dpopt_version": ([], ctypes.c_char_p),
    "dpopt_launch_count": ([], _I64),
    "dpopt_reduce_adamw": ([_PP, _I, _I, _I64, _I, _I64, _P, _P, _P, _P, _F, _F, _F, _F, _I64,
                            _POPT, _P], _I),
    "dpopt_reduce_adamw_buckets": ([_PP, _I, _I, _PI64, _PI64, _I64, _P, _P, _P, _P, _F, _F, _F,
                                    _F, _I64, _POPT, _P], _I),
    "dpopt_grad_sqnorm": ([_PP, _I, _I, _I64, _I, _F, _P, _P, _I64, _P], _I),
    "dpopt_grad_sqnorm_buckets": ([_PP, _I, _I, _PI64, _PI64, _I64, _F, _P, _P, _I64, _P], _I),
    "dpopt_grad_average_sqnorm_buckets": ([_PP, _I, _I, _PI64, _PI64, _I64, _F, _P, _P, _P, _I64,
                                           _P], _I),
    "dpopt_grad_sqnorm_buckets_when_ready": ([_PP, _I, _I, _PI64, _PI64, _I64, _PP, _F, _P, _P, _P,
                                              _I64, _P], _I),
    "dpopt_amp_sqnorm_buckets_when_ready": ([_PP, _I, _I, _PI64, _PI64, _I64, _PP, _P, _P, _P, _P,
                                             _I64, _P], _I),
    "dpopt_grad_sqnorm_scratch_bytes": ([_I64, _I64, _PI64], _I),
    "dpopt_grad_sqnorm_noalloc": ([_PP, _I, _I, _I64, _I, _F, _P, _P], _I),
    "dpopt_grad_average_sqnorm": ([_PP, _I, _I, _I64, _I, _F, _P, _P, _P, _I64, _P], _I),
    "dpopt_loss_scale_init": ([_P, _PCFG, _P], _I),
    "dpopt_amp_sqnorm": ([_PP, _I, _I, _I64, _I, _P, _P, _P, _I64, _P], _I),
    "dpopt_amp_average_sqnorm": ([_PP, _I, _I, _I64, _I, _P, _P, _P, _P, _I64, _P], _I),
    "dpopt_amp_average_sqnorm_buckets": ([_PP, _I, _I, _PI64, _PI64, _I64, _P, _P, _P, _P, _I64,
                                          _P], _I),
    "dpopt_amp_step": ([_PP, _I, _I, _I64, _I, _I64, _P, _P, _P, _P, _F, _F, _F, _F, _F, _F, _P, _P,
                        _PCFG, _P, _P], _I),
    "dpopt_allgather_bf16": ([_P, _I64, _I, _PP, _I, _P], _I),
    "dpopt_reduce_adam_allgather": ([_PP, _I, _I, _I64, _I, _I64, _P, _P, _P, _PP, _F, _F, _F, _F,
                                     _I64, _P], _I),
    "dpopt_reduce_adam_buckets_when_ready": ([_PP, _I, _I, _PI64, _PI64, _I64, _PP, _P, _P, _P,
                                              _P, _F, _F, _F, _F, _I64, _P], _I),
    "dpopt_set_kernel_policy": ([_I], _I),
    "dpopt_get_kernel_policy": ([], _I),
    "dpopt_set_gather_policy": ([_I], _I),
    "dpopt_get_gather_policy": ([], _I),
    "dpopt_selftest_wait_timeout": ([_I64, _P], _I),
    "dpopt_selftest_bounds": ([_P], _I),
}

for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

EXPORTED = tuple(_SIGS)


class DpoptError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.dpopt_last_error().decode(errors="replace")
        name = _lib.dpopt_status_string(status).decode()
        super().__init__(f"{where}: {name}" + (f" ({msg})" if msg else ""))
        self.status = status


def _ptr_array(ptrs: Sequence[int]):
    return (ctypes.c_void_p * len(ptrs))(*ptrs)


# ---------------------------------------------------------------------------
# C ABI, same names
# ---------------------------------------------------------------------------

def dpopt_reduce_adam(grads: Sequence[int], n_replicas: int, numel: int, shard_rank: int,
                      bucket_elems: int, master: int, m: int, v: int, param_bf16_out: int,
                      lr: float, beta1: float, beta2: float, eps: float, step: int,
                      stream: int = 0) -> int:
    return _lib.dpopt_reduce_adam(_ptr_array(grads) if grads is not None else None, n_replicas,
                                  numel, shard_rank, bucket_elems, master, m, v, param_bf16_out,
                                  lr, beta1, beta2, eps, step, stream)


def dpopt_reduce_adam_ex(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                         shard_rank: int, bucket_elems: int, master: int, m: int, v: int,
                         param_bf16_out: int, lr: float, beta1: float, beta2: float, eps: float,
                         step: int, stream: int = 0) -> int:
    return _lib.dpopt_reduce_adam_ex(_ptr_array(grads) if grads is not None else None, grad_dtype,
                                     n_replicas, numel, shard_rank, bucket_elems, master, m, v,
                                     param_bf16_out, lr, beta1, beta2, eps, step, stream)


def dpopt_bucket_count(shard_elems: int, bucket_elems: int) -> tuple[int, int]:
    out = ctypes.c_int64(0)
    rc = _lib.dpopt_bucket_count(shard_elems, bucket_elems, ctypes.byref(out))
    return rc, out.value


def dpopt_bucket_range(shard_elems: int, bucket_elems: int, idx: int) -> tuple[int, int, int]:
    off, ln = ctypes.c_int64(0), ctypes.c_int64(0)
    rc = _lib.dpopt_bucket_range(shard_elems, bucket_elems, idx, ctypes.byref(off),
                                 ctypes.byref(ln))
    return rc, off.value, ln.value


def dpopt_reduce_adam_bucket(grad_slices: Sequence[int], grad_dtype: int, n_replicas: int,
                             shard_offset: int, length: int, master: int, m: int, v: int,
                             param_bf16_out: int, lr: float, beta1: float, beta2: float,
                             eps: float, step: int, stream: int = 0) -> int:
    return _lib.dpopt_reduce_adam_bucket(
        _ptr_array(grad_slices) if grad_slices is not None else None, grad_dtype, n_replicas,
        shard_offset, length, master, m, v, param_bf16_out, lr, beta1, beta2, eps, step, stream)


def dpopt_reduce_adam_buckets(slice_table: Sequence[int], grad_dtype: int, n_replicas: int,
                              offsets: Sequence[int], lens: Sequence[int], master: int, m: int,
                              v: int, param_bf16_out: int, lr: float, beta1: float, beta2: float,
                              eps: float, step: int, stream: int = 0) -> int:
    nb = len(offsets)
    offs = (ctypes.c_int64 * nb)(*offsets)
    lns = (ctypes.c_int64 * nb)(*lens)
    return _lib.dpopt_reduce_adam_buckets(_ptr_array(slice_table), grad_dtype, n_replicas, offs,
                                          lns, nb, master, m, v, param_bf16_out, lr, beta1, beta2,
                                          eps, step, stream)


def dpopt_bucket_table_bytes(n_replicas: int, n_buckets: int) -> tuple[int, int]:
    out = ctypes.c_int64(0)
    rc = _lib.dpopt_bucket_table_bytes(n_replicas, n_buckets, ctypes.byref(out))
    return rc, out.value


def dpopt_reduce_adam_buckets_table(slice_table: Sequence[int], grad_dtype: int, n_replicas: int,
                                    offsets: Sequence[int], lens: Sequence[int], master: int,
                                    m: int, v: int, param_bf16_out: int, lr: float, beta1: float,
                                    beta2: float, eps: float, step: int, opts, table: int,
                                    table_bytes: int, stream: int = 0) -> int:
    nb = len(offsets)
    offs = (ctypes.c_int64 * nb)(*offsets)
    lns = (ctypes.c_int64 * nb)(*lens)
    return _lib.dpopt_reduce_adam_buckets_table(
        _ptr_array(slice_table), grad_dtype, n_replicas, offs, lns, nb, master, m, v,
        param_bf16_out, lr, beta1, beta2, eps, step, _opts(opts), table, table_bytes, stream)


def _opts(opts):
    return ctypes.byref(opts) if opts is not None else None


def dpopt_reduce_adamw(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                       shard_rank: int, bucket_elems: int, master: int, m: int, v: int,
                       param_bf16_out: int, lr: float, beta1: float, beta2: float, eps: float,
                       step: int, opts: StepOptions | None, stream: int = 0) -> int:
    return _lib.dpopt_reduce_adamw(_ptr_array(grads) if grads is not None else None, grad_dtype,
                                   n_replicas, numel, shard_rank, bucket_elems, master, m, v,
                                   param_bf16_out, lr, beta1, beta2, eps, step, _opts(opts),
                                   stream)


def dpopt_reduce_adamw_buckets(slice_table: Sequence[int], grad_dtype: int, n_replicas: int,
                               offsets: Sequence[int], lens: Sequence[int], master: int, m: int,
                               v: int, param_bf16_out: int, lr: float, beta1: float, beta2: float,
                               eps: float, step: int, opts: StepOptions | None,
                               stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_reduce_adamw_buckets(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, master, m, v, param_bf16_out, lr, beta1, beta2, eps,
        step, _opts(opts), stream)


def dpopt_grad_sqnorm(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                      shard_rank: int, grad_unscale: float, sqnorm_out: int, scratch: int,
                      scratch_bytes: int, stream: int = 0) -> int:
    return _lib.dpopt_grad_sqnorm(_ptr_array(grads) if grads is not None else None, grad_dtype,
                                  n_replicas, numel, shard_rank, grad_unscale, sqnorm_out, scratch,
                                  scratch_bytes, stream)


def dpopt_grad_sqnorm_buckets(slice_table: Sequence[int], grad_dtype: int, n_replicas: int,
                              offsets: Sequence[int], lens: Sequence[int], grad_unscale: float,
                              sqnorm_out: int, scratch: int, scratch_bytes: int,
                              stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_grad_sqnorm_buckets(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, grad_unscale, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_grad_average_sqnorm_buckets(slice_table: Sequence[int], grad_dtype: int,
                                      n_replicas: int, offsets: Sequence[int],
                                      lens: Sequence[int], grad_unscale: float, avg_out: int,
                                      sqnorm_out: int, scratch: int, scratch_bytes: int,
                                      stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_grad_average_sqnorm_buckets(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, grad_unscale, avg_out, sqnorm_out, scratch,
        scratch_bytes, stream)


def dpopt_grad_sqnorm_buckets_when_ready(slice_table: Sequence[int], grad_dtype: int,
                                         n_replicas: int, offsets: Sequence[int],
                                         lens: Sequence[int], ready: Sequence[int],
                                         grad_unscale: float, avg_out: int, sqnorm_out: int,
                                         scratch: int, scratch_bytes: int,
                                         stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_grad_sqnorm_buckets_when_ready(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, _ptr_array(ready) if ready is not None else None,
        grad_unscale, avg_out, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_amp_sqnorm_buckets_when_ready(slice_table: Sequence[int], grad_dtype: int,
                                        n_replicas: int, offsets: Sequence[int],
                                        lens: Sequence[int], ready: Sequence[int], state: int,
                                        avg_out: int, sqnorm_out: int, scratch: int,
                                        scratch_bytes: int, stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_amp_sqnorm_buckets_when_ready(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, _ptr_array(ready) if ready is not None else None,
        state, avg_out, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_amp_average_sqnorm_buckets(slice_table: Sequence[int], grad_dtype: int,
                                     n_replicas: int, offsets: Sequence[int], lens: Sequence[int],
                                     state: int, avg_out: int, sqnorm_out: int, scratch: int,
                                     scratch_bytes: int, stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_amp_average_sqnorm_buckets(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, state, avg_out, sqnorm_out, scratch, scratch_bytes,
        stream)


def dpopt_grad_sqnorm_noalloc(grads: Sequence[int], grad_dtype: int, n_replicas: int,
                              numel: int, shard_rank: int, grad_unscale: float, sqnorm_out: int,
                              stream: int = 0) -> int:
    return _lib.dpopt_grad_sqnorm_noalloc(_ptr_array(grads) if grads is not None else None,
                                          grad_dtype, n_replicas, numel, shard_rank, grad_unscale,
                                          sqnorm_out, stream)


def dpopt_grad_average_sqnorm(grads: Sequence[int], grad_dtype: int, n_replicas: int,
                              numel: int, shard_rank: int, grad_unscale: float, avg_out: int,
                              sqnorm_out: int, scratch: int, scratch_bytes: int,
                              stream: int = 0) -> int:
    return _lib.dpopt_grad_average_sqnorm(_ptr_array(grads) if grads is not None else None,
                                          grad_dtype, n_replicas, numel, shard_rank, grad_unscale,
                                          avg_out, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_amp_average_sqnorm(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                             shard_rank: int, state: int, avg_out: int, sqnorm_out: int,
                             scratch: int, scratch_bytes: int, stream: int = 0) -> int:
    return _lib.dpopt_amp_average_sqnorm(_ptr_array(grads) if grads is not None else None,
                                         grad_dtype, n_replicas, numel, shard_rank, state,
                                         avg_out, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_grad_sqnorm_scratch_bytes(elems: int, n_buckets: int = 1) -> tuple[int, int]:
    out = ctypes.c_int64(0)
    rc = _lib.dpopt_grad_sqnorm_scratch_bytes(elems, n_buckets, ctypes.byref(out))
    return rc, out.value


def dpopt_loss_scale_init(state: int, cfg: LossScaleConfig | None, stream: int = 0) -> int:
    return _lib.dpopt_loss_scale_init(state, ctypes.byref(cfg) if cfg is not None else None,
                                      stream)


def dpopt_amp_sqnorm(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                     shard_rank: int, state: int, sqnorm_out: int, scratch: int,
                     scratch_bytes: int, stream: int = 0) -> int:
    return _lib.dpopt_amp_sqnorm(_ptr_array(grads), grad_dtype, n_replicas, numel, shard_rank,
                                 state, sqnorm_out, scratch, scratch_bytes, stream)


def dpopt_amp_step(grads: Sequence[int], grad_dtype: int, n_replicas: int, numel: int,
                   shard_rank: int, bucket_elems: int, master: int, m: int, v: int,
                   param_bf16_out: int, lr: float, beta1: float, beta2: float, eps: float,
                   weight_decay: float, max_grad_norm: float, global_sqnorm: int, state: int,
                   cfg: LossScaleConfig | None, lr_dev: int = 0, stream: int = 0) -> int:
    return _lib.dpopt_amp_step(_ptr_array(grads), grad_dtype, n_replicas, numel, shard_rank,
                               bucket_elems, master, m, v, param_bf16_out, lr, beta1, beta2, eps,
                               weight_decay, max_grad_norm, global_sqnorm, state,
                               ctypes.byref(cfg) if cfg is not None else None, lr_dev, stream)


def dpopt_reduce_adam_buckets_when_ready(slice_table: Sequence[int], grad_dtype: int,
                                         n_replicas: int, offsets: Sequence[int],
                                         lens: Sequence[int], ready: Sequence[int], master: int,
                                         m: int, v: int, param_bf16_out: int, lr: float,
                                         beta1: float, beta2: float, eps: float, step: int,
                                         stream: int = 0) -> int:
    nb = len(offsets)
    return _lib.dpopt_reduce_adam_buckets_when_ready(
        _ptr_array(slice_table), grad_dtype, n_replicas, (ctypes.c_int64 * nb)(*offsets),
        (ctypes.c_int64 * nb)(*lens), nb, _ptr_array(ready), master, m, v, param_bf16_out, lr,
        beta1, beta2, eps, step, stream)


def dpopt_allgather_bf16(shard_bf16: int, shard_elems: int, shard_rank: int,
                         param_replicas: Sequence[int], n_replicas: int, stream: int = 0) -> int:
    return _lib.dpopt_allgather_bf16(shard_bf16, shard_elems, shard_rank,
                                     _ptr_array(param_replicas) if param_replicas is not None
                                     else None, n_replicas, stream)


def dpopt_reduce_adam_allgather(grads: Sequence[int], grad_dtype: int, n_replicas: int,
                                numel: int, shard_rank: int, bucket_elems: int, master: int,
                                m: int, v: int, param_replicas: Sequence[int], lr: float,
                                beta1: float, beta2: float, eps: float, step: int,
                                stream: int = 0) -> int:
    return _lib.dpopt_reduce_adam_allgather(
        _ptr_array(grads) if grads is not None else None, grad_dtype, n_replicas, numel,
        shard_rank, bucket_elems, master, m, v,
        _ptr_array(param_replicas) if param_replicas is not None else None, lr, beta1, beta2,
        eps, step, stream)


def dpopt_stream_status(stream: int = 0) -> int:
    return _lib.dpopt_stream_status(stream)


def dpopt_selftest_bounds(stream: int = 0) -> int:
    return _lib.dpopt_selftest_bounds(stream)


def dpopt_status_string(status: int) -> str:
    return _lib.dpopt_status_string(status).decode()


def dpopt_last_error() -> str:
    return _lib.dpopt_last_error().decode(errors="replace")


def dpopt_state_bytes(psi: int, variant: int, n_dp: int, zero_stage: int) -> tuple[int, float]:
    out = ctypes.c_double(0.0)
    rc = _lib.dpopt_state_bytes(int(psi), variant, n_dp, zero_stage, ctypes.byref(out))
    return rc, out.value


def dpopt_version() -> str:
    return _lib.dpopt_version().decode()


def dpopt_launch_count() -> int:
    return int(_lib.dpopt_launch_count())


def dpopt_set_kernel_policy(policy: int) -> int:
    return _lib.dpopt_set_kernel_policy(policy)


def dpopt_get_kernel_policy() -> int:
    return _lib.dpopt_get_kernel_policy()


def dpopt_set_gather_policy(policy: int) -> int:
    return _lib.dpopt_set_gather_policy(policy)


def dpopt_get_gather_policy() -> int:
    return _lib.dpopt_get_gather_policy()


def dpopt_selftest_wait_timeout(limit_cycles: int, stream: int = 0) -> int:
    return _lib.dpopt_selftest_wait_timeout(limit_cycles, stream)


# ---------------------------------------------------------------------------
# torch-tensor wrappers (marshalling only)
# ---------------------------------------------------------------------------

def _check(rc: int, where: str) -> None:
    if rc != DPOPT_OK:
        raise DpoptError(rc, where)


def _grad_dtype(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DPOPT_GRAD_BF16
    if t.dtype == torch.float32:
        return DPOPT_GRAD_F32
    if t.dtype == torch.float16:
        return DPOPT_GRAD_F16
    raise TypeError(f"gradients must be bfloat16, float16 or float32, got {t.dtype}")


def _operand(t) -> int:
    """The address of a tensor the kernels may read or write: device memory, or
    page-locked host memory (which the device reaches at the same address, so
    the kernels read or write it in place).  Pageable host memory is refused
    here, before any launch, since a kernel could not reach it."""
    if t.is_cuda or t.is_pinned():
        return t.data_ptr()
    raise ValueError("operand is in pageable host memory: move it to the device or pin it "
                     "(pin_memory=True) so that the kernels can address it")


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def reduce_adam(grads, shard_rank: int, bucket_elems: int, master, m, v, param_bf16_out, *,
                lr: float, beta1: float, beta2: float, eps: float, step: int, stream=None) -> None:
    """Full-buffer step: grads are N flattened replica tensors (bf16 or fp32,
    numel elements each); master/m/v (fp32) and param_bf16_out (bf16) hold
    this rank's S = numel/N shard."""
    dt = _grad_dtype(grads[0])
    rc = dpopt_reduce_adam_ex([_operand(g) for g in grads], dt, len(grads), grads[0].numel(),
                              shard_rank, bucket_elems, _operand(master), _operand(m),
                              _operand(v), _operand(param_bf16_out), lr, beta1, beta2, eps, step,
                              _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_ex")


def reduce_adam_bucket(grad_slices, shard_offset: int, master, m, v, param_bf16_out, *, lr: float,
                       beta1: float, beta2: float, eps: float, step: int, stream=None) -> None:
    """One bucket: grad_slices are N tensors of the bucket's length."""
    dt = _grad_dtype(grad_slices[0])
    rc = dpopt_reduce_adam_bucket([_operand(g) for g in grad_slices], dt, len(grad_slices),
                                  shard_offset, grad_slices[0].numel(), _operand(master),
                                  _operand(m), _operand(v), _operand(param_bf16_out), lr, beta1,
                                  beta2, eps, step, _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_bucket")


def reduce_adam_buckets(bucket_slices, offsets, master, m, v, param_bf16_out, *, lr: float,
                        beta1: float, beta2: float, eps: float, step: int, stream=None) -> None:
    """Many buckets: bucket_slices[b] is a list of N tensors for bucket b,
    which updates shard elements [offsets[b], offsets[b] + len)."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    rc = dpopt_reduce_adam_buckets(table, dt, n, list(offsets), lens, _operand(master),
                                   _operand(m), _operand(v), _operand(param_bf16_out), lr,
                                   beta1, beta2, eps, step, _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_buckets")


def bucket_table_bytes(n_replicas: int, n_buckets: int) -> int:
    """Device bytes the one-launch bucket entry needs for its launch table."""
    rc, nbytes = dpopt_bucket_table_bytes(n_replicas, n_buckets)
    _check(rc, "dpopt_bucket_table_bytes")
    return nbytes


def reduce_adam_buckets_table(bucket_slices, offsets, master, m, v, param_bf16_out, table, *,
                              lr: float, beta1: float, beta2: float, eps: float, step: int,
                              opts=None, stream=None) -> None:
    """reduce_adam_buckets in one launch whatever the bucket count: `table` is a
    device tensor of at least bucket_table_bytes(N, len(bucket_slices)) bytes
    that receives the launch table (opts: None for Adam, or step_options())."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    ptrs = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    nbytes = table.numel() * table.element_size()
    rc = dpopt_reduce_adam_buckets_table(ptrs, dt, n, list(offsets), lens, _operand(master),
                                         _operand(m), _operand(v), _operand(param_bf16_out), lr,
                                         beta1, beta2, eps, step, opts, _operand(table), nbytes,
                                         _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_buckets_table")


class BucketStep:
    """The arguments of one batched-bucket call marshalled once: a 274-bucket,
    64-replica list is 17,536 pointers, which take milliseconds to convert on
    every call.  step() then passes the same arrays to
    dpopt_reduce_adam_buckets_table (with `table`: one launch) or to
    dpopt_reduce_adam_buckets (without: launches of at most 2048 pointers).
    The tensors must stay alive and in place while the object is used."""

    def __init__(self, bucket_slices, offsets, master, m, v, param_bf16_out, table=None):
        self.n = len(bucket_slices[0])
        self.dtype = _grad_dtype(bucket_slices[0][0])
        ptrs = [_operand(t) for row in bucket_slices for t in row]
        self.nb = len(bucket_slices)
        self.ptrs = _ptr_array(ptrs)
        self.offs = (ctypes.c_int64 * self.nb)(*offsets)
        self.lens = (ctypes.c_int64 * self.nb)(*[row[0].numel() for row in bucket_slices])
        self.states = [_operand(t) for t in (master, m, v, param_bf16_out)]
        self.table = None if table is None else _operand(table)
        self.table_bytes = 0 if table is None else table.numel() * table.element_size()

    def step(self, *, lr: float, beta1: float, beta2: float, eps: float, step: int, opts=None,
             stream=None) -> None:
        st = _stream_handle(stream)
        if self.table is not None:
            rc = _lib.dpopt_reduce_adam_buckets_table(
                self.ptrs, self.dtype, self.n, self.offs, self.lens, self.nb, *self.states, lr,
                beta1, beta2, eps, step, _opts(opts), self.table, self.table_bytes, st)
            _check(rc, "dpopt_reduce_adam_buckets_table")
        elif opts is not None:
            rc = _lib.dpopt_reduce_adamw_buckets(self.ptrs, self.dtype, self.n, self.offs,
                                                 self.lens, self.nb, *self.states, lr, beta1,
                                                 beta2, eps, step, _opts(opts), st)
            _check(rc, "dpopt_reduce_adamw_buckets")
        else:
            rc = _lib.dpopt_reduce_adam_buckets(self.ptrs, self.dtype, self.n, self.offs,
                                                self.lens, self.nb, *self.states, lr, beta1,
                                                beta2, eps, step, st)
            _check(rc, "dpopt_reduce_adam_buckets")


def step_options(weight_decay: float = 0.0, max_grad_norm: float = 0.0, grad_sqnorm=None,
                 grad_unscale: float = 0.0) -> StepOptions:
    """Build a dpopt_step_options; grad_sqnorm is a 1-element float64 device tensor."""
    return StepOptions(weight_decay, max_grad_norm,
                       _operand(grad_sqnorm) if grad_sqnorm is not None else None, grad_unscale)


def reduce_adamw(grads, shard_rank: int, bucket_elems: int, master, m, v, param_bf16_out, *,
                 lr: float, beta1: float, beta2: float, eps: float, step: int,
                 opts: StepOptions | None, stream=None) -> None:
    dt = _grad_dtype(grads[0])
    rc = dpopt_reduce_adamw([_operand(g) for g in grads], dt, len(grads), grads[0].numel(),
                            shard_rank, bucket_elems, _operand(master), _operand(m), _operand(v),
                            _operand(param_bf16_out), lr, beta1, beta2, eps, step, opts,
                            _stream_handle(stream))
    _check(rc, "dpopt_reduce_adamw")


def reduce_adamw_buckets(bucket_slices, offsets, master, m, v, param_bf16_out, *, lr: float,
                         beta1: float, beta2: float, eps: float, step: int,
                         opts: StepOptions | None, stream=None) -> None:
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    rc = dpopt_reduce_adamw_buckets(table, dt, n, list(offsets), lens, _operand(master),
                                    _operand(m), _operand(v), _operand(param_bf16_out), lr,
                                    beta1, beta2, eps, step, opts, _stream_handle(stream))
    _check(rc, "dpopt_reduce_adamw_buckets")


def grad_sqnorm(grads, shard_rank: int, sqnorm_out, scratch, *, grad_unscale: float = 0.0,
                stream=None) -> None:
    """sqnorm_out: 1-element float64 device tensor; scratch: device tensor of at least
    dpopt_grad_sqnorm_scratch_bytes(S) bytes."""
    dt = _grad_dtype(grads[0])
    rc = dpopt_grad_sqnorm([_operand(g) for g in grads], dt, len(grads), grads[0].numel(),
                           shard_rank, grad_unscale, _operand(sqnorm_out), _operand(scratch),
                           scratch.numel() * scratch.element_size(), _stream_handle(stream))
    _check(rc, "dpopt_grad_sqnorm")


def grad_average_sqnorm(grads, shard_rank: int, avg_out, sqnorm_out, scratch, *,
                        grad_unscale: float = 0.0, stream=None) -> None:
    """grad_sqnorm that also writes the shard's fixed-order average gradient to
    avg_out (float32 device tensor of S = numel / N elements)."""
    dt = _grad_dtype(grads[0])
    rc = dpopt_grad_average_sqnorm([_operand(g) for g in grads], dt, len(grads),
                                   grads[0].numel(), shard_rank, grad_unscale, _operand(avg_out),
                                   _operand(sqnorm_out), _operand(scratch),
                                   scratch.numel() * scratch.element_size(),
                                   _stream_handle(stream))
    _check(rc, "dpopt_grad_average_sqnorm")


def amp_average_sqnorm(grads, shard_rank: int, state, avg_out, sqnorm_out, scratch,
                       stream=None) -> None:
    dt = _grad_dtype(grads[0])
    rc = dpopt_amp_average_sqnorm([_operand(g) for g in grads], dt, len(grads),
                                  grads[0].numel(), shard_rank, _operand(state),
                                  _operand(avg_out), _operand(sqnorm_out), _operand(scratch),
                                  scratch.numel() * scratch.element_size(), _stream_handle(stream))
    _check(rc, "dpopt_amp_average_sqnorm")


def grad_sqnorm_buckets(bucket_slices, offsets, sqnorm_out, scratch, *, grad_unscale: float = 0.0,
                        stream=None) -> None:
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    rc = dpopt_grad_sqnorm_buckets(table, dt, n, list(offsets), lens, grad_unscale,
                                   _operand(sqnorm_out), _operand(scratch),
                                   scratch.numel() * scratch.element_size(), _stream_handle(stream))
    _check(rc, "dpopt_grad_sqnorm_buckets")


def grad_average_sqnorm_buckets(bucket_slices, offsets, avg_out, sqnorm_out, scratch, *,
                                grad_unscale: float = 0.0, stream=None) -> None:
    """grad_sqnorm_buckets that also writes each element's fixed-order average
    to avg_out at its shard offset (float32 device tensor indexed like the
    states); the buckets must continue one another (contiguous gradients)."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    rc = dpopt_grad_average_sqnorm_buckets(table, dt, n, list(offsets), lens, grad_unscale,
                                           _operand(avg_out), _operand(sqnorm_out),
                                           _operand(scratch),
                                           scratch.numel() * scratch.element_size(),
                                           _stream_handle(stream))
    _check(rc, "dpopt_grad_average_sqnorm_buckets")


def amp_average_sqnorm_buckets(bucket_slices, offsets, state, avg_out, sqnorm_out, scratch, *,
                               stream=None) -> None:
    """amp_sqnorm over bucket slices that continue one another, storing each
    element's average at its shard offset (the step then reads avg_out)."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    rc = dpopt_amp_average_sqnorm_buckets(table, dt, n, list(offsets), lens, _operand(state),
                                          _operand(avg_out), _operand(sqnorm_out),
                                          _operand(scratch),
                                          scratch.numel() * scratch.element_size(),
                                          _stream_handle(stream))
    _check(rc, "dpopt_amp_average_sqnorm_buckets")


def loss_scale_init(state, init_scale: float = 65536.0, window: int = 1000, hysteresis: int = 2,
                    min_scale: float = 1.0, stream=None) -> LossScaleConfig:
    """state: a device tensor of at least 32 bytes (e.g. torch.zeros(4, dtype=torch.int64)).
    Returns the config to pass to amp_step."""
    cfg = LossScaleConfig(init_scale, window, hysteresis, min_scale)
    _check(dpopt_loss_scale_init(_operand(state), cfg, _stream_handle(stream)),
           "dpopt_loss_scale_init")
    return cfg


def read_loss_scale(state) -> LossScaleState:
    """Copy the device state to the host (synchronises)."""
    raw = state.detach().cpu().numpy().tobytes()[:ctypes.sizeof(LossScaleState)]
    return LossScaleState.from_buffer_copy(raw)


def amp_sqnorm(grads, shard_rank: int, state, sqnorm_out, scratch, stream=None) -> None:
    dt = _grad_dtype(grads[0])
    rc = dpopt_amp_sqnorm([_operand(g) for g in grads], dt, len(grads), grads[0].numel(),
                          shard_rank, _operand(state), _operand(sqnorm_out), _operand(scratch),
                          scratch.numel() * scratch.element_size(), _stream_handle(stream))
    _check(rc, "dpopt_amp_sqnorm")


def amp_step(grads, shard_rank: int, bucket_elems: int, master, m, v, param_bf16_out, *,
             lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
             max_grad_norm: float, global_sqnorm, state, cfg: LossScaleConfig,
             lr_dev=None, stream=None) -> None:
    """lr_dev: None, or a float32 device tensor holding the learning rate, read
    when the step runs (lr is then not used)."""
    dt = _grad_dtype(grads[0])
    rc = dpopt_amp_step([_operand(g) for g in grads], dt, len(grads), grads[0].numel(),
                        shard_rank, bucket_elems, _operand(master), _operand(m), _operand(v),
                        _operand(param_bf16_out), lr, beta1, beta2, eps, weight_decay,
                        max_grad_norm, 0 if global_sqnorm is None else _operand(global_sqnorm),
                        _operand(state), cfg, 0 if lr_dev is None else _operand(lr_dev),
                        stream=_stream_handle(stream))
    _check(rc, "dpopt_amp_step")


def reduce_adam_buckets_when_ready(bucket_slices, offsets, ready_events, master, m, v,
                                  param_bf16_out, *, lr: float, beta1: float, beta2: float,
                                  eps: float, step: int, stream=None) -> None:
    """ready_events: one torch.cuda.Event (already recorded) or None per bucket."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    ready = [e.cuda_event if e is not None else 0 for e in ready_events]
    rc = dpopt_reduce_adam_buckets_when_ready(table, dt, n, list(offsets), lens, ready,
                                              _operand(master), _operand(m), _operand(v),
                                              _operand(param_bf16_out), lr, beta1, beta2, eps,
                                              step, _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_buckets_when_ready")


def grad_sqnorm_buckets_when_ready(bucket_slices, offsets, ready_events, sqnorm_out, scratch, *,
                                   avg_out=None, grad_unscale: float = 0.0,
                                   stream=None) -> None:
    """The norm pass bucket by bucket behind each bucket's event (one
    torch.cuda.Event or None per bucket); avg_out (float32 device tensor indexed
    like the states) also receives each element's average."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    ready = [e.cuda_event if e is not None else 0 for e in ready_events]
    rc = dpopt_grad_sqnorm_buckets_when_ready(table, dt, n, list(offsets), lens, ready,
                                              grad_unscale,
                                              0 if avg_out is None else _operand(avg_out),
                                              _operand(sqnorm_out), _operand(scratch),
                                              scratch.numel() * scratch.element_size(),
                                              _stream_handle(stream))
    _check(rc, "dpopt_grad_sqnorm_buckets_when_ready")


def amp_sqnorm_buckets_when_ready(bucket_slices, offsets, ready_events, state, sqnorm_out,
                                  scratch, *, avg_out=None, stream=None) -> None:
    """grad_sqnorm_buckets_when_ready with the unscale 1/scale read from the
    device loss-scale state."""
    n = len(bucket_slices[0])
    dt = _grad_dtype(bucket_slices[0][0])
    table = [_operand(t) for row in bucket_slices for t in row]
    lens = [row[0].numel() for row in bucket_slices]
    ready = [e.cuda_event if e is not None else 0 for e in ready_events]
    rc = dpopt_amp_sqnorm_buckets_when_ready(table, dt, n, list(offsets), lens, ready,
                                             _operand(state),
                                             0 if avg_out is None else _operand(avg_out),
                                             _operand(sqnorm_out), _operand(scratch),
                                             scratch.numel() * scratch.element_size(),
                                             _stream_handle(stream))
    _check(rc, "dpopt_amp_sqnorm_buckets_when_ready")


def allgather_bf16(shard_bf16, shard_rank: int, param_replicas, stream=None) -> None:
    """Write the bf16 shard tensor into every replica's flat bf16 parameter tensor
    at the shard's position."""
    rc = dpopt_allgather_bf16(_operand(shard_bf16), shard_bf16.numel(), shard_rank,
                              [_operand(t) for t in param_replicas], len(param_replicas),
                              _stream_handle(stream))
    _check(rc, "dpopt_allgather_bf16")


def reduce_adam_allgather(grads, shard_rank: int, bucket_elems: int, master, m, v,
                          param_replicas, *, lr: float, beta1: float, beta2: float, eps: float,
                          step: int, stream=None) -> None:
    """The full-buffer step with the bf16 shard written into every replica's
    flat parameter tensor (param_replicas[shard_rank] holds the working copy)."""
    dt = _grad_dtype(grads[0])
    rc = dpopt_reduce_adam_allgather([_operand(g) for g in grads], dt, len(grads),
                                     grads[0].numel(), shard_rank, bucket_elems,
                                     _operand(master), _operand(m), _operand(v),
                                     [_operand(t) for t in param_replicas], lr, beta1, beta2,
                                     eps, step, _stream_handle(stream))
    _check(rc, "dpopt_reduce_adam_allgather")


def stream_status(stream=None) -> None:
    _check(dpopt_stream_status(_stream_handle(stream)), "dpopt_stream_status")


class kernel_policy:
    """Context manager: run the enclosed calls with a given kernel policy."""

    def __init__(self, policy: int):
        self.policy = policy

    def __enter__(self):
        self.saved = dpopt_get_kernel_policy()
        _check(dpopt_set_kernel_policy(self.policy), "dpopt_set_kernel_policy")
        return self

    def __exit__(self, *exc):
        dpopt_set_kernel_policy(self.saved)
        return False


class gather_policy:
    """Context manager: run the enclosed calls with a given all-gather form."""

    def __init__(self, policy: int):
        self.policy = policy

    def __enter__(self):
        self.saved = dpopt_get_gather_policy()
        _check(dpopt_set_gather_policy(self.policy), "dpopt_set_gather_policy")
        return self

    def __exit__(self, *exc):
        dpopt_set_gather_policy(self.saved)
        return False
