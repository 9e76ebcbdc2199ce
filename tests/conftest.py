import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_terminal_summary(terminalreporter):
    """One line per floating-point parity comparison of the run: the plain
    max|err| / RMS(y_ref) next to the tolerance and the asserted excess over
    the bf16 flip allowance (tests/gpu_util.py)."""
    try:
        from tests.gpu_util import PARITY_LOG
    except Exception:
        return
    if not PARITY_LOG:
        return
    terminalreporter.section("parity: max|err|/RMS per comparison")
    for what, st in PARITY_LOG:
        terminalreporter.write_line(
            f"{what:<40s} max|err|/RMS {st['max_err_over_rms']:.3e}  "
            f"excess/RMS {st['max_excess_over_rms']:.3e}  rms_err/RMS "
            f"{st['rms_err_over_rms']:.3e}  tol {st['tol']:g}  n {st['n']}")
