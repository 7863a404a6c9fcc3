import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Table of the elements that met the tolerance only against the bf16-operand
    emulation (few-key edge cases), so that the count shows even under ``-q``."""
    try:
        from gpu_util import FALLBACK_LOG
    except Exception:
        return
    if not FALLBACK_LOG:
        return
    tr = terminalreporter
    n_cmp = len(FALLBACK_LOG)
    used = [r for r in FALLBACK_LOG if r[1] > 0]
    tr.write_sep("-", "oracle parity: elements outside the tolerance that only the bf16 emulation accepts")
    tr.write_line(f"{n_cmp} comparisons against the oracle; {n_cmp - len(used)} with no such element")
    for what, n, size, frac in used:
        tr.write_line(f"  {what}: {n} of {size} elements (cap {int(frac * size)})")
