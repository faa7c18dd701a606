"""Shared pytest set-up: the ``gpu`` marker, the repo root on ``sys.path``, and
lazily built native libraries (the oracle on any host, the product library
only for GPU tests and the symbol/validation checks)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def psk_lib():
    """The product C-ABI library, built if missing (cross-compiles without a GPU)."""
    from paged_sparse_kv_gb300 import build as psk_build
    psk_build.build()
    from paged_sparse_kv_gb300 import _abi
    return _abi.lib()


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_sparse_kv_gb300 import build as psk_build
    psk_build.build()
    return torch.device("cuda:0")
