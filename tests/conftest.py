import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size workloads)")


def pytest_terminal_summary(terminalreporter):
    """The largest per-step errors seen against the oracle, per configuration
    (in units of the oracle value's ulp; err/tol is against 2.4e-7 x scale)."""
    mod = sys.modules.get("tests.parity")
    log = getattr(mod, "ULP_LOG", None)
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "per-step parity against the oracle (max over checked values)")
    tr.write_line(f"{'configuration':44s} {'checks':>6s} {'ulp master':>10s} {'ulp m':>7s} "
                  f"{'ulp v':>7s} {'err/tol':>8s} {'bitwise':>8s}")
    for name in sorted(log):
        n, um, umm, uv, et, bw = log[name]
        tr.write_line(f"{name[:44]:44s} {n:6d} {um:10.2f} {umm:7.2f} {uv:7.2f} {et:8.3f} "
                      f"{bw:8.5f}")
