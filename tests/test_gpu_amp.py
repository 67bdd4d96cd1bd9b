"""fp16 gradients and the loss-scaled step (the fp16 block of the ZeRO-3
answer's DeepSpeed config) on the GPU against the oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import parity
from tests.parity import grad_host_range, oracle_amp_trajectory, oracle_trajectory

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import zero_mixed_precision_gb300 as dp
    from tests.test_gpu_parity import _run_small_full, _small_workload, f32, to_dev_grad, u16
else:
    dp = None

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 13, 64])
@pytest.mark.parametrize("S", [7, 4097, 100_003])
def test_fp16_gradients_every_element(n, S):
    _need_gpu()
    wl = _small_workload(n, S, kind=2)
    refs = oracle_trajectory(wl, np.arange(S), 1, 2)
    got = _run_small_full(wl, steps=(1, 2))
    parity.check(refs[-1], *got, where=f"fp16 N={n} S={S}")


def _amp_workload(n, S):
    # scaled fp16 gradients: N(0, 1e-3) times a nominal 2^10, outliers x100
    return synth.Workload(name="amp", n_replicas=n, numel=n * S, shard_rank=1, bucket_elems=S,
                          seed=41, grad_dist=lambda r: synth.Dist(0.0, 1.0, 0.01, 100.0),
                          master_dist=synth.Dist(0.0, 0.02), m_dist=None, v_dist=None, steps=1,
                          grad_kind=2)


@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_loss_scaled_run_with_overflows_matches_the_oracle(max_norm):
    """Ten iterations, window 3, hysteresis 2: overflows injected at iterations
    4, 6, 7 (an Inf in another rank's part of one replica) skip the step, move the
    scale and hold the step count, on the device exactly as in the oracle."""
    _need_gpu()
    n, S = 4, 20_000
    wl = _amp_workload(n, S)
    inject = {4: (2, 3 * S + 11, 0x7C00), 6: (0, 5, 0xFC00), 7: (3, S - 1, 0x7E00)}

    def full(k):
        bufs = [grad_host_range(wl, r, k, 0, wl.numel) for r in range(n)]
        if k in inject:
            r, i, bits = inject[k]
            bufs[r][i] = bits
        return bufs

    cfg_args = dict(init_scale=1024.0, window=3, hysteresis=2, min_scale=1.0)
    refs = oracle_amp_trajectory(wl, 10, full, oracle.LossScaler(1024.0, 3, 2, 1.0),
                                 weight_decay=0.01, max_grad_norm=max_norm)

    master, m, v = parity.states_host(wl, wl.shard_base + np.arange(S))
    dm, dmm, dv = (torch.from_numpy(x.copy()).cuda() for x in (master, m, v))
    dout = torch.zeros(S, dtype=torch.bfloat16, device="cuda")
    state = torch.zeros(4, dtype=torch.int64, device="cuda")
    cfg = dp.loss_scale_init(state, **cfg_args)
    rc, nbytes = dp.dpopt_grad_sqnorm_scratch_bytes(S, 1)
    scratch = torch.empty(nbytes // 8, dtype=torch.float64, device="cuda")
    part = torch.zeros(n, dtype=torch.float64, device="cuda")
    total = torch.zeros(1, dtype=torch.float64, device="cuda")
    for k in range(1, 11):
        prev = (f32(dm), f32(dmm), f32(dv))
        host = full(k)
        grads = [to_dev_grad(b) for b in host]
        for r in range(n):   # every rank's norm; their sum is the one-scalar all-reduce
            dp.amp_sqnorm(grads, r, state, part[r:r + 1], scratch)
        torch.sum(part, dim=0, keepdim=True, out=total)
        dp.amp_step(grads, wl.shard_rank, S, dm, dmm, dv, dout, weight_decay=0.01,
                    max_grad_norm=max_norm, global_sqnorm=total, state=state, cfg=cfg, **HP)
        dp.stream_status()
        st = dp.read_loss_scale(state)
        ref, overflow, scale, steps = refs[k - 1]
        assert bool(st.last_overflow) == overflow, k
        assert (st.scale, st.step) == (scale, steps), (k, st.scale, st.step, scale, steps)
        if steps > 0:
            got = (f32(dm), f32(dmm), f32(dv), u16(dout))
            parity.check(ref, *got, where=f"amp k={k}")
        if not overflow:
            # this iteration's step on its own, from the GPU's previous states
            un = 1.0 / refs[k - 2][2] if k > 1 else 1.0 / cfg_args["init_scale"]
            c = oracle.grad_scale(oracle.grad_sqnorm(host, 0, wl.numel, un), max_norm, un)
            base = wl.shard_base
            parity.check_step(wl, np.arange(S), steps, prev, got, f"amp fp16 N={n} S={S}",
                              grads_fn=lambda r, _t: host[r][base:base + S], weight_decay=0.01,
                              gscale_fn=lambda _t, _g: c)
    assert st.skipped == 3


def test_amp_entry_points_validate_their_arguments():
    _need_gpu()
    state = torch.zeros(4, dtype=torch.int64, device="cuda")
    bad = dp.LossScaleConfig(0.0, 1000, 2, 1.0)
    assert dp.dpopt_loss_scale_init(state.data_ptr(), bad, 0) == dp.DPOPT_ERR_INVALID_ARG
    bad = dp.LossScaleConfig(1024.0, 0, 2, 1.0)
    assert dp.dpopt_loss_scale_init(state.data_ptr(), bad, 0) == dp.DPOPT_ERR_INVALID_ARG
    ok = dp.LossScaleConfig(1024.0, 10, 2, 1.0)
    assert dp.dpopt_loss_scale_init(state.data_ptr() + 4, ok, 0) == dp.DPOPT_ERR_INVALID_ARG
    assert dp.dpopt_loss_scale_init(state.data_ptr(), ok, 0) == dp.DPOPT_OK
    dp.stream_status()
    st = dp.read_loss_scale(state)
    assert (st.scale, st.good_steps, st.hysteresis_left, st.step, st.skipped) == (1024.0, 0, 2, 0, 0)
