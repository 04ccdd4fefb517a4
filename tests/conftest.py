import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst max-relative output errors per workload seen by the GPU parity checks (tests/_gpu.py WORST)."""
    g = sys.modules.get("tests._gpu")
    worst = getattr(g, "WORST", None) if g is not None else None
    if not worst:
        return
    tr = terminalreporter
    tr.write_sep("-", "worst max-relative output error per workload")
    tr.write_line(f"{'workload':56s} {'vs rounded':>11s} {'vs exact':>10s} {'beyond 1 rnd':>12s} {'rows':>8s}")
    for label in sorted(worst):
        w = worst[label]
        tr.write_line(f"{label:56s} {w['rounded']:11.3e} {w['exact_nonrope']:10.3e} {w['beyond_rounding']:12.3e} "
                      f"{w['rows']:8d}")
    tr.write_line("vs rounded: all dims, against the oracle rounded at the pages' storage points; vs exact: non-rope "
                  "dims against the un-rounded oracle; beyond 1 rnd: the same less half an ulp of each element")
