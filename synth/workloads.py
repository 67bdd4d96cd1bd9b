"""Workload recipes: sizes, value distributions and seeds of the synthetic
inputs.  Data only -- no arithmetic of the method.

Sizes follow the workloads the method is specified on: a flat buffer the
size of GPT-2 small (124M parameters), a 1.3B-parameter flat buffer, one
rank's ZeRO-3 shard of a 70B model at 64-way data parallelism, plus a tiny
case and a size sweep.  No weights or datasets exist or are needed: "124M",
"1.3B" and "70B" are sizes only, and every value is drawn from the seeded
generator of this package.

Streams: stream id = (kind << 56) | (replica << 32) | step, kinds below.  A
gradient value is indexed by its position in the flattened replica buffer; a
state value (master, m, v) by its position in the flattened parameter vector,
so the shards of different ranks of one model are slices of one vector.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Optional

STREAM_GRAD = 1
STREAM_MASTER = 2
STREAM_M = 3
STREAM_V = 4


def stream_id(kind: int, replica: int = 0, step: int = 0) -> int:
    assert 0 <= kind < 256 and 0 <= replica < (1 << 24) and 0 <= step < (1 << 32)
    return (kind << 56) | (replica << 32) | step


@dataclass(frozen=True)
class Dist:
    """x = mu + sigma*z (z ~ Irwin-Hall(12) normal); with probability outlier_p
    x *= outlier_scale; |x| when absval."""
    mu: float = 0.0
    sigma: float = 1.0
    outlier_p: float = 0.0
    outlier_scale: float = 1.0
    absval: bool = False


@dataclass(frozen=True)
class Workload:
    name: str
    n_replicas: int
    numel: int                  # elements of one flattened replica buffer
    shard_rank: int
    bucket_elems: int
    seed: int
    grad_dist: Callable[[int], Dist]      # replica -> distribution
    master_dist: Dist
    m_dist: Optional[Dist]                # None: zeros
    v_dist: Optional[Dist]
    steps: int                            # measured Adam steps
    warmup_steps: int = 0                 # steps run before the measured ones
    grad_kind: int = 0                    # 0 bf16, 1 fp32, 2 fp16
    layout: str = "full"                  # "full": N full buffers; "slices": N shard slices
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    note: str = field(default="")

    @property
    def shard_elems(self) -> int:
        return self.numel // self.n_replicas

    @property
    def shard_base(self) -> int:
        return self.shard_rank * self.shard_elems

    def grad_bytes(self) -> int:
        return 4 if self.grad_kind == 1 else 2

    def bytes_per_param(self) -> int:
        # N gradient reads + master/m/v read and write (24) + bf16 write (2)
        return self.grad_bytes() * self.n_replicas + 26

    def first_step(self) -> int:
        return self.warmup_steps + 1


def _const(d: Dist) -> Callable[[int], Dist]:
    return lambda r: d


WORKLOADS: dict[str, Workload] = {
    # N=2, one 4096-element shard, single bucket, 3 steps, seed 0
    "tiny": Workload(
        name="tiny", n_replicas=2, numel=8192, shard_rank=0, bucket_elems=4096, seed=0,
        grad_dist=_const(Dist(0.0, 1e-3)), master_dist=Dist(0.0, 0.02), m_dist=None, v_dist=None,
        steps=3),
    # GPT-2-small-sized flat buffer: 124M, N=4, rank 0 (31M), 25M buckets + 6M tail,
    # 1% of entries x100 (outliers), 10 steps
    "gpt2s": Workload(
        name="gpt2s", n_replicas=4, numel=124_000_000, shard_rank=0, bucket_elems=25_000_000,
        seed=1, grad_dist=_const(Dist(0.0, 1e-3, outlier_p=0.01, outlier_scale=100.0)),
        master_dist=Dist(0.0, 0.02), m_dist=None, v_dist=None, steps=10),
    # 1.3B flat buffer, N=8, rank 3 (162.5M), 50M buckets + 12.5M tail, per-replica
    # bias k*1e-5, 5 pre-warm steps then 5 measured steps
    "1p3b": Workload(
        name="1p3b", n_replicas=8, numel=1_300_000_000, shard_rank=3, bucket_elems=50_000_000,
        seed=2, grad_dist=lambda r: Dist(r * 1e-5, 1e-4), master_dist=Dist(0.0, 0.02),
        m_dist=None, v_dist=None, steps=5, warmup_steps=5),
    # one rank's ZeRO-3 shard of a 70B model at N=64: 1.09375e9 params, 4M-element
    # buckets (273 full + 1.75M tail), 64 replica slices resident, 2 steps
    "70b_shard": Workload(
        name="70b_shard", n_replicas=64, numel=70_000_000_000, shard_rank=0,
        bucket_elems=4_000_000, seed=3, grad_dist=_const(Dist(0.0, 1e-4)),
        master_dist=Dist(0.0, 0.02), m_dist=Dist(0.0, 1e-4), v_dist=Dist(0.0, 1e-8, absval=True),
        steps=2, layout="slices"),
}

SWEEP_SIZES = (1_000_000, 16_000_000, 256_000_000, 1_000_000_000)
SWEEP_REPLICAS = (1, 2, 8, 32, 64)


def sweep_cell(shard_elems: int, n_replicas: int, grad_kind: int) -> Workload:
    """One cell of the size sweep: N slices of S elements each (a single
    bucket), values ~ N(0, 1e-3), master ~ N(0, 0.02), m = v = 0, one step."""
    return Workload(
        name=f"sweep_S{shard_elems}_N{n_replicas}_{'bf16' if grad_kind == 0 else 'f32'}",
        n_replicas=n_replicas, numel=shard_elems * n_replicas, shard_rank=0,
        bucket_elems=shard_elems, seed=4, grad_dist=_const(Dist(0.0, 1e-3)),
        master_dist=Dist(0.0, 0.02), m_dist=None, v_dist=None, steps=1, grad_kind=grad_kind,
        layout="slices")
