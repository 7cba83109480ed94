import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmx")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


def pytest_terminal_summary(terminalreporter):
    """Observed GEMM accuracy of the parity tests that ran: the worst error
    as a fraction of the allowed bound and as a fraction of T = sum |a*b|,
    per test file and output type; and the incident-trace counts (clipped,
    zeroed values, NaN/Inf blocks) read off GPU-quantized tensors."""
    from mxcheck import ERROR_LOG, INCIDENT_LOG
    if INCIDENT_LOG:
        terminalreporter.write_sep("-", "incident-trace counts of GPU-quantized tensors")
        for test, what, n, clipped, zeroed, nan_blocks in INCIDENT_LOG:
            terminalreporter.write_line(
                f"{what}: {n} values, {clipped} clipped, {zeroed} zeroed, "
                f"{nan_blocks} NaN/Inf blocks")
    if not ERROR_LOG:
        return
    worst = {}
    for test, dtype, ratio, rel_t, n in ERROR_LOG:
        key = (test.split("::")[0], dtype)
        w = worst.setdefault(key, [0.0, 0.0, 0])
        w[0] = max(w[0], ratio)
        w[1] = max(w[1], rel_t)
        w[2] += n
    terminalreporter.write_sep("-", "observed GEMM accuracy (max over checked outputs)")
    for (path, dtype), (ratio, rel_t, n) in sorted(worst.items()):
        terminalreporter.write_line(
            f"{path} {dtype}: error/bound {ratio:.3g}, max |y - y_ref| / T {rel_t:.3g}, "
            f"{n} outputs")
