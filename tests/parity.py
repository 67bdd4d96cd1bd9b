"""Parity harness: seeded inputs for the oracle and the CUDA path, the oracle's
trajectory on (sampled) elements, and the tolerance check.

Tolerance (the required bound: fp32 master/m/v within 2.4e-7 relative, ~2 ulp; bf16
output within 1 bf16 ulp).  "Relative" is taken against the scale of the
terms each stored value is formed from, so that cancellation does not turn
one rounding into many ulps:
  m:      scale_m = max(|beta1*m_prev|, |(1-beta1)*g|, |m_new|)
  v:      scale_v = v_new                      (all terms >= 0)
  master: scale_t = max(|theta_prev|, |theta_new|, |delta|, delta~), where
          delta~ = a*M/D is the update with |m_new| replaced by the m scale
          accumulated so far (a = lr/bc1, D = sqrt(v_new/bc2) + eps): the
          part of the master that a difference in m can move.
Two checks use these scales:
  per step (the stated bound): the oracle runs step t alone from the GPU's
      own states after step t-1, and every value of step t must lie within
      2.4e-7 times that step's scale (check_step);
  trajectory: the oracle runs every step from the initial states; a
      difference left by step t carries into step t+1, so step t is checked
      against 2.4e-7 times the sum of the scales of steps 1..t.
Both floor the allowance at FLT_MIN.  bf16: ordered-integer distance <= 1,
and the GPU's bf16 must equal RNE(its own master) exactly.  Every per-step
check records its largest errors (in ulps of the oracle's value) under its
configuration's name; the test session prints them at the end.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synth
from synth import Workload, stream_id, STREAM_GRAD, STREAM_MASTER, STREAM_M, STREAM_V

REL_TOL = 2.4e-7
FLT_MIN = float(np.finfo(np.float32).tiny)


# ---------------------------------------------------------------------------
# inputs
# ---------------------------------------------------------------------------

def _typed(wl: Workload, a: np.ndarray) -> np.ndarray:
    return oracle.as_f16_bits(a) if wl.grad_kind == synth.KIND_F16 else a


def grad_host(wl: Workload, r: int, t: int, idx: np.ndarray) -> np.ndarray:
    """Replica r's gradient of step t at flattened replica-buffer indices idx."""
    return _typed(wl, synth.host_gather(wl.grad_kind, idx, wl.seed,
                                        stream_id(STREAM_GRAD, r, t), wl.grad_dist(r)))


def grad_host_range(wl: Workload, r: int, t: int, start: int, count: int) -> np.ndarray:
    return _typed(wl, synth.host_fill(wl.grad_kind, start, count, wl.seed,
                                      stream_id(STREAM_GRAD, r, t), wl.grad_dist(r)))


def states_host(wl: Workload, gidx: np.ndarray):
    """Initial master, m, v at flattened parameter indices gidx."""
    master = synth.host_gather(1, gidx, wl.seed, stream_id(STREAM_MASTER), wl.master_dist)
    m = (synth.host_gather(1, gidx, wl.seed, stream_id(STREAM_M), wl.m_dist)
         if wl.m_dist is not None else np.zeros(gidx.size, np.float32))
    v = (synth.host_gather(1, gidx, wl.seed, stream_id(STREAM_V), wl.v_dist)
         if wl.v_dist is not None else np.zeros(gidx.size, np.float32))
    return master, m, v


# ---------------------------------------------------------------------------
# oracle trajectory with tolerance scales
# ---------------------------------------------------------------------------

@dataclass
class StepRef:
    t: int
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    out: np.ndarray
    tol_master: np.ndarray
    tol_m: np.ndarray
    tol_v: np.ndarray


def _f64(x):
    return np.asarray(x, dtype=np.float64)


class _Tolerance:
    """Running tolerance allowances of one trajectory (see the module doc)."""

    def __init__(self, size: int, hp: dict):
        self.b1 = float(np.float32(hp["beta1"]))
        self.b2 = float(np.float32(hp["beta2"]))
        self.lr = float(np.float32(hp["lr"]))
        self.eps = float(np.float32(hp["eps"]))
        self.acc_m = np.zeros(size)
        self.acc_v = np.zeros(size)
        self.acc_t = np.zeros(size)

    def step(self, t, g, th_prev, m_prev, master, m, v):
        b1, b2, lr, eps = self.b1, self.b2, self.lr, self.eps
        bc1 = 1.0 - b1 ** t
        bc2 = 1.0 - b2 ** t
        scale_m = np.maximum.reduce([np.abs(b1 * m_prev), np.abs((1.0 - b1) * _f64(g)),
                                     np.abs(_f64(m))])
        self.acc_m += scale_m
        self.acc_v += _f64(v)
        with np.errstate(all="ignore"):
            D = np.sqrt(_f64(v) / bc2) + eps
            a = lr / bc1
            delta = a * _f64(m) / D
            delta_m = a * self.acc_m / D
            delta_v = np.abs(delta) * self.acc_v / np.maximum(2.0 * _f64(v), FLT_MIN)
        scale_t = np.maximum.reduce([np.abs(th_prev), np.abs(_f64(master)), np.abs(delta),
                                     delta_m, np.minimum(delta_v, np.abs(delta) * 8)])
        scale_t = np.where(np.isfinite(scale_t), scale_t, 0.0)
        self.acc_t += scale_t

    def ref(self, t, master, m, v, out) -> "StepRef":
        return StepRef(t, master.copy(), m.copy(), v.copy(), out,
                       REL_TOL * np.maximum(self.acc_t, FLT_MIN),
                       REL_TOL * np.maximum(self.acc_m, FLT_MIN),
                       REL_TOL * np.maximum(self.acc_v, FLT_MIN))


def oracle_trajectory(wl: Workload, local_idx: np.ndarray, t_first: int, t_last: int,
                      grads_fn=None, init=None, hp=None, weight_decay: float = 0.0,
                      gscale_fn=None) -> list[StepRef]:
    """Run the oracle over steps t_first..t_last on the shard elements local_idx
    (0 <= j < S) and return every step's states and tolerances.

    grads_fn(r, t) -> gradient values at those elements (default: the seeded
    generator at flattened index shard_base + j); init -> (master, m, v)
    (default: the seeded generator).  weight_decay: AdamW decay; gscale_fn(t,
    grads) -> the fp32 gradient multiplier of step t (clipping / unscaling),
    computed by the oracle from that step's gradients."""
    hp = hp or dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    gidx = wl.shard_base + np.asarray(local_idx, dtype=np.int64)
    if grads_fn is None:
        def grads_fn(r, t):
            return grad_host(wl, r, t, gidx)
    master, m, v = init if init is not None else states_host(wl, gidx)
    master, m, v = master.copy(), m.copy(), v.copy()
    tol = _Tolerance(master.size, hp)
    refs = []
    for t in range(t_first, t_last + 1):
        grads = [grads_fn(r, t) for r in range(wl.n_replicas)]
        g = oracle.average(grads)
        if gscale_fn is not None:
            c = np.float32(gscale_fn(t, grads))
            g = (_f64(g) * np.float64(c)).astype(np.float32)
        th_prev, m_prev = _f64(master), _f64(m)
        out = oracle.adam(g, master, m, v, step=t, weight_decay=weight_decay, **hp)
        tol.step(t, g, th_prev, m_prev, master, m, v)
        refs.append(tol.ref(t, master, m, v, out))
    return refs


def oracle_amp_trajectory(wl: Workload, iters: int, full_grads_fn, scaler, *,
                          weight_decay: float = 0.0, max_grad_norm: float = 0.0, hp=None):
    """Loss-scaled run of the oracle over every element of the shard: at each
    iteration k (1-based) full_grads_fn(k) gives the N whole replica buffers
    (scaled gradients); the oracle decides overflow from the global norm,
    skips or steps, and advances the scaler.  Returns per iteration
    (StepRef, overflow, scale_after, optimizer_steps_after)."""
    hp = hp or dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps)
    S, base = wl.shard_elems, wl.shard_base
    master, m, v = states_host(wl, base + np.arange(S, dtype=np.int64))
    tol = _Tolerance(S, hp)
    out = oracle.f32_to_bf16(master)
    res = []
    for k in range(1, iters + 1):
        full = full_grads_fn(k)
        unscale = 1.0 / scaler.scale
        sq = oracle.grad_sqnorm(full, 0, full[0].size, unscale)
        overflow = not np.isfinite(sq)
        if not overflow:
            c = oracle.grad_scale(sq, max_grad_norm, unscale)
            g = (_f64(oracle.average([x[base:base + S] for x in full])) * np.float64(c)).astype(
                np.float32)
            th_prev, m_prev = _f64(master), _f64(m)
            t = scaler.step + 1
            out = oracle.adam(g, master, m, v, step=t, weight_decay=weight_decay, **hp)
            tol.step(t, g, th_prev, m_prev, master, m, v)
        scaler.update(overflow)
        res.append((tol.ref(scaler.step, master, m, v, out), overflow, scaler.scale, scaler.step))
    return res


# ---------------------------------------------------------------------------
# comparison
# ---------------------------------------------------------------------------

def bf16_ordered(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def _same_nonfinite(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise: both NaN, or both the same infinity."""
    a64, b64 = _f64(a), _f64(b)
    return (np.isnan(a64) & np.isnan(b64)) | (np.isinf(a64) & (a64 == b64))


@dataclass
class Stats:
    n: int
    max_ulp_master: float
    max_ulp_m: float
    max_ulp_v: float
    max_err_over_tol: float
    bitwise_master: float
    bitwise_out: float


def check(ref: StepRef, master, m, v, out, where: str = "") -> Stats:
    """Assert GPU values (numpy arrays at the same elements) match ref."""
    master = np.asarray(master, np.float32)
    m = np.asarray(m, np.float32)
    v = np.asarray(v, np.float32)
    out = np.asarray(out).view(np.uint16) if np.asarray(out).dtype != np.uint16 else np.asarray(out)
    worst = 0.0
    ulps = []
    for name, got, want, tol in (("master", master, ref.master, ref.tol_master),
                                 ("m", m, ref.m, ref.tol_m), ("v", v, ref.v, ref.tol_v)):
        fin = np.isfinite(want)
        bad_nf = ~fin & ~_same_nonfinite(got, want)
        assert not bad_nf.any(), (
            f"{where} step {ref.t} {name}: non-finite mismatch at {np.flatnonzero(bad_nf)[:5]}")
        err = np.abs(_f64(got[fin]) - _f64(want[fin]))
        assert np.all(np.isfinite(got[fin])), f"{where} step {ref.t} {name}: finite expected"
        ratio = err / tol[fin] if err.size else np.zeros(0)
        if ratio.size and ratio.max() > 1.0:
            k = int(np.argmax(ratio))
            j = np.flatnonzero(fin)[k]
            raise AssertionError(
                f"{where} step {ref.t} {name}[{j}]: gpu {got[j]!r} oracle {want[j]!r} "
                f"err {err[k]:.3e} > tol {tol[j]:.3e}")
        worst = max(worst, float(ratio.max()) if ratio.size else 0.0)
        spacing = np.spacing(np.abs(want[fin])).astype(np.float64)
        ulps.append(float((err / np.maximum(spacing, 1e-45)).max()) if err.size else 0.0)
    # bf16: within one ulp of the oracle's, and exactly RNE of the GPU's own master
    d = np.abs(bf16_ordered(out) - bf16_ordered(ref.out))
    fin_out = np.isfinite(oracle.bf16_to_f64(ref.out))
    assert np.all(d[fin_out] <= 1), f"{where} step {ref.t} bf16 off by {d[fin_out].max()} ulp"
    own = oracle.f32_to_bf16(master)
    nan_own = np.isnan(oracle.bf16_to_f64(own))
    assert np.array_equal(out[~nan_own], own[~nan_own]), f"{where}: bf16 != RNE(own master)"
    assert np.all(np.isnan(oracle.bf16_to_f64(out[nan_own]))), f"{where}: NaN master -> NaN bf16"
    return Stats(int(master.size), ulps[0], ulps[1], ulps[2], worst,
                 float(np.mean(master.view(np.uint32) == ref.master.view(np.uint32))),
                 float(np.mean(out == ref.out)))


# ---------------------------------------------------------------------------
# per-step check: one oracle step from the GPU's own previous states
# ---------------------------------------------------------------------------

# configuration -> [checks, max ulp master, m, v, max err/tol, min bitwise master]
ULP_LOG: dict[str, list] = {}


def record(config: str, st: Stats) -> None:
    e = ULP_LOG.setdefault(config, [0, 0.0, 0.0, 0.0, 0.0, 1.0])
    e[0] += 1
    e[1] = max(e[1], st.max_ulp_master)
    e[2] = max(e[2], st.max_ulp_m)
    e[3] = max(e[3], st.max_ulp_v)
    e[4] = max(e[4], st.max_err_over_tol)
    e[5] = min(e[5], st.bitwise_master)


def check_step(wl: Workload, local_idx: np.ndarray, t: int, prev, got, config: str,
               grads_fn=None, hp=None, weight_decay: float = 0.0, gscale_fn=None) -> Stats:
    """Step t on its own: the oracle starts from prev = (master, m, v), the
    GPU's states at local_idx after step t-1, and got = (master, m, v, bf16)
    after step t must match within 2.4e-7 times step t's scales (one step's
    allowance, nothing carried over) and 1 bf16 ulp."""
    init = tuple(np.array(x, dtype=np.float32, copy=True) for x in prev)
    ref = oracle_trajectory(wl, local_idx, t, t, grads_fn=grads_fn, init=init, hp=hp,
                            weight_decay=weight_decay, gscale_fn=gscale_fn)[0]
    st = check(ref, *got, where=f"{config} (step {t} alone)")
    record(config, st)
    return st
