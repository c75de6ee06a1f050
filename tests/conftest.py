import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def orc():
    """The fp64 oracle (compiled from oracle/gsi_oracle.c on first use)."""
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def gsi():
    """The CUDA library binding; fails loudly if it cannot load on a GPU machine."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_rank_subspace_gsi_gb300 import lib
    return lib
