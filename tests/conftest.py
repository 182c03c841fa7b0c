import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of CPU)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


def _cuda_ok():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when selected without a GPU: a GPU test
    # run that silently skipped would look green.
    pass


@pytest.fixture(scope="session")
def gpu():
    """The built library and torch on cuda:0; GPU tests depend on this."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    import ordered_merge_gb300 as om

    return om


@pytest.fixture(params=["default", "ring"])
def merge_path(request, monkeypatch):
    """Runs a merge test twice: with the library's own choice of kernel
    (merges that fit in one wave take the one-pass kernel) and with the
    circular-buffer tile-merge kernel forced for every size."""
    if request.param == "ring":
        monkeypatch.setenv("OM_ONE_PASS_MAX", "0")
    else:
        monkeypatch.delenv("OM_ONE_PASS_MAX", raising=False)
    return request.param
