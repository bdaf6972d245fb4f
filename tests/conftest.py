import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path through the C-ABI)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_terminal_summary(terminalreporter):
    """Print the largest bf16 error ratio each GPU parity test saw (the
    relative bound's margin), when any were recorded."""
    mod = sys.modules.get("gpu_harness")
    ratios = getattr(mod, "RATIOS", None)
    if not ratios:
        return
    terminalreporter.write_sep("-", "bf16: largest max|gpu - oracle| / (2^-8 max|oracle|) per test")
    for name, r in sorted(ratios.items(), key=lambda kv: -kv[1]):
        terminalreporter.write_line(f"{r:7.3f}  {name}")
