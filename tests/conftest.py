import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(autouse=True)
def _cuda_core_opt_in(request, monkeypatch):
    """The parity tests also cover the bf16 shapes that only the CUDA-core
    kernels take, which the library runs only on request; the tests of that
    refusal remove the variable again."""
    if "gpu" in request.keywords:
        monkeypatch.setenv("CAAT_ALLOW_FALLBACK", "1")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
