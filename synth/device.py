"""Device-resident workload buffers filled by the seeded generator.

Allocation (torch) and filling (synth_dev.cu) only; no arithmetic of the
method.  Shared by the GPU tests and the benchmark.
"""
from __future__ import annotations

import torch

import synth
from synth import Workload, stream_id, STREAM_GRAD, STREAM_MASTER, STREAM_M, STREAM_V

BF16_NAN = 0x7FC0


class DeviceWorkload:
    """Buffers of one workload on one device.

    layout "full": N flattened replica buffers of numel elements; the rank's
    shard [base, base+S) of each holds seeded gradients, everything outside it
    holds NaN, so a read outside the shard poisons the result.
    layout "slices": N buffers of S elements (the rank's slice of each replica)."""

    def __init__(self, wl: Workload, device: str | torch.device = "cuda:0"):
        self.wl = wl
        self.device = torch.device(device)
        S, n = wl.shard_elems, wl.n_replicas
        gdt = {0: torch.bfloat16, 1: torch.float32, 2: torch.float16}[wl.grad_kind]
        glen = wl.numel if wl.layout == "full" else S
        self.grads = [torch.empty(glen, dtype=gdt, device=self.device) for _ in range(n)]
        if wl.layout == "full":
            for g in self.grads:
                g.fill_(float("nan"))
        self.master = torch.empty(S, dtype=torch.float32, device=self.device)
        self.m = torch.empty(S, dtype=torch.float32, device=self.device)
        self.v = torch.empty(S, dtype=torch.float32, device=self.device)
        self.out = torch.empty(S, dtype=torch.bfloat16, device=self.device)

    # -- filling -----------------------------------------------------------------
    def _stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def fill_states(self) -> None:
        wl, S = self.wl, self.wl.shard_elems
        base = wl.shard_base
        synth.device_fill(self.master.data_ptr(), 1, base, S, wl.seed, stream_id(STREAM_MASTER),
                          wl.master_dist, self._stream())
        for buf, kind, dist in ((self.m, STREAM_M, wl.m_dist), (self.v, STREAM_V, wl.v_dist)):
            if dist is None:
                buf.zero_()
            else:
                synth.device_fill(buf.data_ptr(), 1, base, S, wl.seed, stream_id(kind), dist,
                                  self._stream())
        self.out.view(torch.int16).fill_(BF16_NAN)

    def fill_grads(self, t: int) -> None:
        """Step t's gradients of every replica (the rank's shard range only)."""
        wl, S = self.wl, self.wl.shard_elems
        esize = wl.grad_bytes()
        off = wl.shard_base if wl.layout == "full" else 0
        for r, g in enumerate(self.grads):
            synth.device_fill(g.data_ptr() + off * esize, wl.grad_kind, wl.shard_base, S, wl.seed,
                              stream_id(STREAM_GRAD, r, t), wl.grad_dist(r), self._stream())

    # -- views -------------------------------------------------------------------
    def shard_slices(self) -> list[torch.Tensor]:
        """Each replica's view of the rank's shard."""
        wl = self.wl
        if wl.layout == "full":
            return [g[wl.shard_base:wl.shard_base + wl.shard_elems] for g in self.grads]
        return list(self.grads)

    def bucket_slices(self, bucket_elems: int | None = None):
        """[(shard_offset, [N slice views])] for every bucket of the shard."""
        be = bucket_elems or self.wl.bucket_elems
        S = self.wl.shard_elems
        sl = self.shard_slices()
        out = []
        for off in range(0, S, be):
            ln = min(be, S - off)
            out.append((off, [s[off:off + ln] for s in sl]))
        return out

    def bytes_resident(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   [*self.grads, self.master, self.m, self.v, self.out])


def workload_bytes(wl: Workload) -> int:
    """Device bytes a DeviceWorkload of wl allocates."""
    glen = wl.numel if wl.layout == "full" else wl.shard_elems
    return wl.n_replicas * glen * wl.grad_bytes() + wl.shard_elems * 14
