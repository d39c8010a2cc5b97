import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 GPU and the built CUDA library (run with -m gpu)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report how many GEMM/BMM outputs met the 2-ulp bar only under the
    fp32-summation allowance (the tolerance reading for near-cancelling sums)."""
    try:
        from helpers import ALLOWANCE_LOG
    except ImportError:
        return
    if not ALLOWANCE_LOG:
        return
    n = sum(r["n"] for r in ALLOWANCE_LOG)
    n_allow = sum(r["n_allowance"] for r in ALLOWANCE_LOG)
    small = [r for r in ALLOWANCE_LOG if r["K"] is not None and r["K"] <= 512]
    worst = max(r["max_ulp"] for r in ALLOWANCE_LOG if r["n_allowance"] == 0) if any(
        r["n_allowance"] == 0 for r in ALLOWANCE_LOG) else None
    tr = terminalreporter
    tr.write_line(f"parity: {len(ALLOWANCE_LOG)} oracle comparisons, {n} outputs; {n_allow} within 2 ulp only "
                  f"under the fp32-summation allowance; K <= 512 comparisons: {len(small)} with "
                  f"{sum(r['n_allowance'] for r in small)} such outputs; largest error of the comparisons that "
                  f"needed none: {worst:.2f} ulp" if worst is not None else "")
    for r in ALLOWANCE_LOG:
        if r["n_allowance"]:
            tr.write_line(f"  allowance used: {r['n_allowance']} of {r['n']} outputs in {r['what'] or '?'} "
                          f"(K={r['K']})")
