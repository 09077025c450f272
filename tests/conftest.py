import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The loaded C-ABI library; GPU tests fail (not skip) if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_decode_step_weight_gb300 import api
    return api.lib()


# Measured parity figures (errors, agreement counts) recorded by the GPU tests;
# written as JSON to $QD_PARITY_LOG at the end of the session when that is set.
_PARITY = {}


@pytest.fixture(scope="session")
def parity_log():
    return _PARITY


def pytest_sessionfinish(session, exitstatus):
    path = os.environ.get("QD_PARITY_LOG")
    if path and _PARITY:
        with open(path, "w") as f:
            json.dump(_PARITY, f, indent=1, sort_keys=True)
