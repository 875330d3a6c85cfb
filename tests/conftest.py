import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device visible: GPU parity tests need the GB300")
    return torch.device("cuda:0")


# One line per parity test that logs its comparison (tolerance accounting:
# exact fraction, largest error in ulps, values beyond one ulp, e4m3 codes,
# exponent near-ties), printed at the end of the run.
_PARITY_LOG = []


@pytest.fixture
def parity_log(request):
    def log(*reports):
        _PARITY_LOG.append(f"{request.node.name}: " + " | ".join(r.summary() for r in reports))
    return log


def pytest_terminal_summary(terminalreporter):
    if _PARITY_LOG:
        terminalreporter.section("parity against the oracle")
        for line in _PARITY_LOG:
            terminalreporter.write_line(line)
