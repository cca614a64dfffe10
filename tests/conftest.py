import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU work")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def kda():
    """The CUDA library's Python binding; loading fails loudly if it is not built."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kda_delta_rule_fwd_gb300 as m
    m.load()  # raises if the shared library is missing
    return m
