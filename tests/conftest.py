import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU oracle runs")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every oracle comparison's error (max abs, relative L2) against the tolerance."""
    try:
        import gpu_harness
    except Exception:
        return
    if not gpu_harness.PARITY_LOG:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the fp64 oracle (tolerance: max abs 2e-2, rel L2 5e-3)")
    for test, mx, rel in gpu_harness.PARITY_LOG:
        tr.write_line(f"{test}: max_abs {mx:.3e} rel_l2 {rel:.3e}")
