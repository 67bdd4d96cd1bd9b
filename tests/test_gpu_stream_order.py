"""Stream order holds across the library's programmatic dependent launches:
every library kernel may be scheduled while the kernel before it on the
stream is still running, and waits for it (griddepcontrol.wait) before its
first memory access.  A chain of producer kernels (PyTorch's), steps, norm
passes and consumers on one stream with no host synchronisation must give
bit for bit what the same chain gives with a full synchronisation between
every call."""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _chain(sync: bool):
    n, S = 4, 8_000_003
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    src = [torch.randn(n * S, generator=gen, device="cuda").mul_(1e-3).bfloat16()
           for _ in range(n)]
    master = torch.randn(S, generator=gen, device="cuda").mul_(0.02)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    out = torch.empty(S, dtype=torch.bfloat16, device="cuda")
    # the gradient buffers start as NaN: a step that ran ahead of its producer
    # would read them
    grads = [torch.full((n * S,), float("nan"), dtype=torch.bfloat16, device="cuda")
             for _ in range(n)]
    avg = torch.empty(S, device="cuda")
    sq = torch.zeros(1, dtype=torch.float64, device="cuda")
    scratch = torch.empty(dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)[1] // 8 + 1,
                          dtype=torch.float64, device="cuda")
    opts = dp.step_options(weight_decay=0.01, max_grad_norm=0.5, grad_sqnorm=sq)
    keep = []

    def fence():
        if sync:
            torch.cuda.synchronize()

    torch.cuda.synchronize()
    for t in (1, 2, 3):
        for g, s in zip(grads, src):      # producer: a PyTorch copy and scale
            g.copy_(s)
            g.mul_(1.0 + t / 8)
        fence()
        dp.reduce_adam(grads, 1, S, master, m, v, out, step=t, **HP)
        fence()
        keep.append(out.float().sum())    # consumer: a PyTorch reduction of the output
        fence()
        dp.grad_average_sqnorm(grads, 1, avg, sq, scratch)
        fence()
        dp.reduce_adamw([avg], 0, S, master, m, v, out, step=t + 3, opts=opts, **HP)
        fence()
        keep.append(out.float().sum())
    torch.cuda.synchronize()
    assert dp.dpopt_stream_status(0) == 0
    return [x.cpu().numpy() for x in (master, m, v, out.view(torch.int16), avg, sq)] + \
        [np.array([k.item() for k in keep])]


def test_unsynchronised_chain_equals_the_synchronised_one():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a = _chain(sync=False)
    b = _chain(sync=True)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert np.isfinite(a[0]).all() and np.isfinite(a[-1]).all()
