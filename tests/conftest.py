import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_dev():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """GEMM parity records: per check, the elements that needed the bf16 half-ulp
    term and the worst |err| / bound with and without it."""
    try:
        import gpu_util
    except Exception:
        return
    if not gpu_util.RECORDS:
        return
    tr = terminalreporter
    tr.section("GEMM tolerance records")
    tot_n = tot_used = 0
    worst_plain = 0.0
    for test, tol in gpu_util.RECORDS:
        tr.write_line("%-90s %r" % (test[-90:], tol))
        tot_n += tol.n
        tot_used += tol.half_ulp_used
        worst_plain = max(worst_plain, tol.worst_plain)
    tr.write_line("all checks: %d elements, %d needed the half-ulp term, worst |err|/bound without it %.3g"
                  % (tot_n, tot_used, worst_plain))
