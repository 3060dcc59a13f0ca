import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_terminal_summary(terminalreporter):
    from . import report
    if not report.QUANT_ERRORS:
        return
    tr = terminalreporter
    tr.write_sep("-", "quantization error of Y against the unquantized fp64 X W^T (+ LoRA)")
    for name, rows, rel, mx, ref in report.QUANT_ERRORS:
        tr.write_line(f"{name:<28} rows {rows:5d}  rel L2 {rel:.4f}  max |err| {mx:.3f}  "
                      f"(max |Y| {ref:.1f})")
