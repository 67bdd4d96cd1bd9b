"""Fused ZeRO gradient reduce + mixed-precision Adam for one GB300 (sm_103a).

The compute path is libdpopt.so (hand-written CUDA, C ABI in include/dpopt.h);
this package is its ctypes binding.  Importing it without the built library
fails loudly; there is no CPU or PyTorch fallback.
"""
from .binding import *  # noqa: F401,F403
from .binding import (  # noqa: F401
    DpoptError, EXPORTED, LIB_PATH, LossScaleConfig, allgather_bf16, LossScaleState, StepOptions, amp_sqnorm,
    amp_average_sqnorm, grad_average_sqnorm,
    amp_step, gather_policy, grad_sqnorm, grad_sqnorm_buckets, kernel_policy, loss_scale_init,
    read_loss_scale,
    reduce_adam, reduce_adam_allgather, reduce_adam_bucket, reduce_adam_buckets,
    reduce_adam_buckets_when_ready,
    reduce_adamw, reduce_adamw_buckets,
    step_options, stream_status,
)

__version__ = "0.1.0"
