import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_100-family) and the built kernel library")


def pytest_terminal_summary(terminalreporter):
    """Per configuration: the worst O and LSE errors of the GPU parity checks,
    with the mean O error against the unrounded fp64 result beside the one
    against it rounded to bf16 (the asserted one)."""
    try:
        from tests.gpu_util import PARITY_LOG
    except ImportError:
        return
    if not PARITY_LOG:
        return
    worst = {}
    for cfg, _label, mx, mean_b, mean_x, el in PARITY_LOG:
        w = worst.setdefault(cfg, [0.0, 0.0, 0.0, 0.0, 0])
        w[0] = max(w[0], mx)
        w[1] = max(w[1], mean_b)
        w[2] = max(w[2], mean_x)
        w[3] = max(w[3], el)
        w[4] += 1
    tr = terminalreporter
    tr.write_line("parity vs fp64 oracle (worst over checks): config | max|dO| | "
                  "mean|dO-bf16(O)| | mean|dO| exact | max|dLSE| | checks")
    for cfg, (mx, mb, mx_, el, n) in worst.items():
        tr.write_line(f"  {cfg} | {mx:.3e} | {mb:.3e} | {mx_:.3e} | {el:.3e} | {n}")
