import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes on the CPU oracle)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def fno():
    """The CUDA library binding; builds the shared library first if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fft_gemm_ifft_gb300 import build as fbuild
    fbuild.build()
    import fft_gemm_ifft_gb300 as pkg
    return pkg
