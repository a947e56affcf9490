import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture
def tune():
    """Sets the library's tuning overrides for one test (forge_set_tuning) and
    restores the previous ones afterwards.  Fields not given keep their value."""
    from weight_gradient_gemm_gb300 import _build
    from weight_gradient_gemm_gb300 import forge as F
    _build.build()
    saved = F.get_tuning()

    def set_(**kw):
        F.set_tuning(**{**F.get_tuning(), **kw})

    yield set_
    F.set_tuning(**saved)
