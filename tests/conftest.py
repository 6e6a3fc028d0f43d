import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()


@pytest.fixture(params=["1", "2"], ids=["cta1", "cta2"])
def gemm_kernel(request, monkeypatch):
    """Run a tensor-core test once with the one-CTA GEMM and once with the
    CTA-pair GEMM (TPS_GEMM_KERNEL is read at every launch)."""
    monkeypatch.setenv("TPS_GEMM_KERNEL", request.param)
    return request.param
