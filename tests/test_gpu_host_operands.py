"""Host-resident operands: gradients in page-locked host memory read in place
by the step kernel, and the bf16 working copy written straight into
page-locked host memory.  The results must equal, bit for bit, those of the
same call on device-resident copies (the arithmetic does not depend on where
an operand lives), and match the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth
from synth.device import DeviceWorkload
from tests import parity
from tests.parity import oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import f32, u16
else:
    dp = None


def _wl(layout: str):
    # a ragged shard (not a multiple of 8) over several buckets
    return synth.Workload(name="host_operands", n_replicas=4, numel=4 * 1_000_003, shard_rank=1,
                          bucket_elems=300_000, seed=61,
                          grad_dist=lambda r: synth.Dist(0.0, 1e-3),
                          master_dist=synth.Dist(0.0, 0.02), m_dist=None, v_dist=None, steps=2,
                          layout=layout)


def _pinned_like(t: torch.Tensor) -> torch.Tensor:
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


def _clone_states(dev):
    return dev.master.clone(), dev.m.clone(), dev.v.clone()


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    return np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("layout", ["slices", "full"])
def test_host_gradients_and_host_output_equal_the_device_call(layout):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _wl(layout)
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    dev = DeviceWorkload(wl)
    dev.fill_states()
    torch.cuda.synchronize()
    runs = {}
    states = {k: _clone_states(dev) for k in ("device", "host")}
    outs = {"device": torch.empty_like(dev.out),
            "host": torch.empty(dev.out.shape, dtype=torch.bfloat16, pin_memory=True)}
    rng = np.random.default_rng(9)
    idx = np.unique(np.concatenate([rng.integers(0, wl.shard_elems, 20_000),
                                    np.arange(wl.shard_elems - 50, wl.shard_elems)]))
    for t in (1, 2):
        prev = [f32(x)[idx] for x in states["host"]]
        dev.fill_grads(t)
        torch.cuda.synchronize()
        host_grads = [_pinned_like(g) for g in dev.grads]
        for kind, grads in (("device", dev.grads), ("host", host_grads)):
            th, m, v = states[kind]
            if layout == "full":
                dp.reduce_adam(grads, wl.shard_rank, wl.bucket_elems, th, m, v, outs[kind],
                               step=t, **hp)
            else:
                dp.reduce_adam_bucket(grads, 0, th, m, v, outs[kind], step=t, **hp)
        torch.cuda.synchronize()
        dp.stream_status()
        got = [f32(x)[idx] for x in states["host"]] + [u16(outs["host"])[idx]]
        parity.check_step(wl, idx, t, prev, got, f"host operands ({layout})")
    for kind in ("device", "host"):
        th, m, v = states[kind]
        runs[kind] = [f32(th), f32(m), f32(v), u16(outs[kind])]
    for a, b in zip(runs["device"], runs["host"]):
        assert _same(a, b)
    refs = oracle_trajectory(wl, idx, 1, 2)
    parity.check(refs[-1], *(x[idx] for x in runs["host"]), where=f"host operands ({layout})")


def test_misaligned_host_slices_equal_the_device_call():
    """Host slices that start 4 bytes past a 16-byte boundary take the scalar
    head and then the vector body, as device slices do."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = _wl("slices")
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, step=1)
    dev = DeviceWorkload(wl)
    dev.fill_states()
    dev.fill_grads(1)
    torch.cuda.synchronize()
    S = wl.shard_elems
    res = []
    for where in ("device", "host"):
        th, m, v = _clone_states(dev)
        if where == "device":
            bufs = [torch.empty(S + 1, dtype=g.dtype, device=g.device) for g in dev.grads]
            out = torch.zeros(S, dtype=torch.bfloat16, device=dev.master.device)
        else:
            bufs = [torch.empty(S + 1, dtype=g.dtype, pin_memory=True) for g in dev.grads]
            out = torch.zeros(S, dtype=torch.bfloat16).pin_memory()
        for b, g in zip(bufs, dev.grads):
            b[1:].copy_(g)
        # elements 1 .. S-1 of the shard: the slices start 4 bytes past a
        # 16-byte boundary, the states and the output at shard offset 1
        dp.reduce_adam_bucket([b[2:] for b in bufs], 1, th, m, v, out, **hp)
        torch.cuda.synchronize()
        dp.stream_status()
        res.append([f32(th), f32(m), f32(v), u16(out)])
    for a, b in zip(*res):
        assert _same(a, b)
