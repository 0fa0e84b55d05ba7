import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """fp32 parity held to the TF32 bound: how many elements of each case lie
    beyond the fp32 tolerance pair atol 1e-3 / rtol 1e-2."""
    try:
        from gpu_util import TF32_RECORDS
    except Exception:
        return
    if not TF32_RECORDS:
        return
    terminalreporter.write_sep("-", "fp32 (TF32) parity: elements beyond atol 1e-3 / rtol 1e-2, all within the TF32 bound")
    for what, beyond, n, worst in TF32_RECORDS:
        terminalreporter.write_line(f"{what}: {beyond} of {n} beyond atol 1e-3 / rtol 1e-2; worst err/bound {worst:.3f}")
