"""The oracle's pins are sensitive: plant one plausible mistake at a time in a
copy of the oracle's C source (on the CPU), rebuild it, and check that at
least one pin of tests/test_oracle_pins.py fails on the mutant."""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "update sign flipped": ("th - delta", "th + delta"),
    "(1-beta1) dropped": ("(1.0 - h->beta1) * g", "g"),
    "g instead of g^2 in v": ("(1.0 - h->beta2) * g * g", "(1.0 - h->beta2) * g"),
    "bias-correction index off by one": ("h.bc1 = 1.0 - pow(h.beta1, (double)step);",
                                         "h.bc1 = 1.0 - pow(h.beta1, (double)step + 1.0);"),
    "betas swapped in bias correction": ("h.bc1 = 1.0 - pow(h.beta1,", "h.bc1 = 1.0 - pow(h.beta2,"),
    "eps inside the sqrt": ("sqrt(v_hat) + h->eps", "sqrt(v_hat + h->eps)"),
    "m_hat not bias-corrected": ("double m_hat = (double)m32 / h->bc1;", "double m_hat = (double)m32;"),
    "fp32 replica accumulation": ("    double s = 0.0;\n    for (int r = 0;",
                                  "    float s = 0.0f;\n    for (int r = 0;"),
    "1/N dropped": ("(double)s32 / (double)n", "(double)s32"),
    "replica 0 skipped": ("for (int r = 0; r < n; ++r)", "for (int r = 1; r < n; ++r)"),
    "bf16 ties away from zero": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "bf16 truncation": ("lower > 0x8000u ||", "0 &&"),
    "weight decay on the new theta": ("h->lr * h->weight_decay * th;",
                                      "h->lr * h->weight_decay * (th - delta);"),
    "clip coefficient not clamped to 1": ("if (coef < 1.0) c *= coef;", "c *= coef;"),
    "clip on the squared norm": ("max_norm / (sqrt(sqnorm) + 1e-6);", "max_norm / (sqnorm + 1e-6);"),
    "unscale not applied in the norm": ("* (double)unscale;\n        acc += x * x;",
                                        ";\n        acc += x * x;"),
}

PIN_FUNCS = [
    (pins.test_bf16_rne_matches_torch_cpu_library_rounding, {}),
    (pins.test_average_equals_exact_rational_average_bruteforce, {"n": 3}),
    (pins.test_average_equals_exact_rational_average_bruteforce, {"n": 1}),
    (pins.test_identical_replicas_average_to_the_input_exactly, {"n": 8}),
    (pins.test_cancellation_keeps_the_small_term, {}),
    (pins.test_adam_matches_torch_optim_adam_float64,
     {"hp": dict(lr=1e-2, b1=0.8, b2=0.95, eps=1e-3)}),
    (pins.test_adamw_matches_torch_optim_adamw_float64, {}),
    (pins.test_first_step_closed_form, {}),
    (pins.test_constant_gradient_closed_form, {}),
    (pins.test_sqnorm_matches_exact_rational_sum_of_squares, {}),
    (pins.test_clipping_matches_torch_clip_grad_norm, {}),
]


def _load(path):
    saved = oracle._lib
    oracle._lib = None
    real = oracle._LIB_PATH
    oracle._LIB_PATH = path
    try:
        L = oracle.lib()
    finally:
        oracle._LIB_PATH = real
        oracle._lib = saved
    return L


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation anchor must occur exactly once: {old!r}"
    mutant_c = tmp_path / "oracle_mutant.c"
    mutant_c.write_text(src.replace(old, new, 1), encoding="utf-8")
    so = tmp_path / "liboracle_mutant.so"
    cmd = oracle.build_command()
    cmd[cmd.index(SRC)] = str(mutant_c)
    cmd[cmd.index(oracle._LIB_PATH)] = str(so)
    subprocess.run(cmd, check=True)
    mutant = _load(str(so))
    saved = oracle._lib
    oracle._lib = mutant
    failures = 0
    try:
        for fn, kw in PIN_FUNCS:
            try:
                fn(**kw)
            except AssertionError:
                failures += 1
    finally:
        oracle._lib = saved
    assert failures >= 1, f"no pin caught the planted mistake: {name}"


# The accounting lives in the oracle's Python part: each mutant below replaces
# state_components with a plausible misreading of the ZeRO stages, and at least
# one golden accounting row must fail on it.
def _stage_mutant(shard_p_from, shard_g_from, shard_o_from):
    real = oracle.state_components

    def mutant(psi, variant, n_dp, zero_stage):
        c = real(psi, variant, 1, 0)   # the unsharded components
        return {"params": c["params"] / (n_dp if zero_stage >= shard_p_from else 1),
                "grads": c["grads"] / (n_dp if zero_stage >= shard_g_from else 1),
                "optimizer": c["optimizer"] / (n_dp if zero_stage >= shard_o_from else 1)}
    return mutant


@pytest.mark.parametrize("name,stages", [
    ("gradients sharded from stage 1", (3, 1, 1)),
    ("optimizer sharded only from stage 2", (3, 2, 2)),
    ("parameters sharded from stage 2", (2, 2, 1)),
    ("stages shifted by one", (2, 1, 0)),
])
def test_planted_accounting_mistake_is_caught(name, stages, monkeypatch):
    monkeypatch.setattr(oracle, "state_components", _stage_mutant(*stages))
    failures = 0
    for row in pins._golden_rows():
        try:
            pins.test_state_accounting_matches_printed_figures(row)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"no golden accounting row caught: {name}"
