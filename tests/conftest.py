import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True, scope="module")
def _device_error_word_stays_clear():
    """After every module that loaded the library on a GPU: no kernel may have
    given up on a bounded wait (the per-device error word stays 0)."""
    yield
    mod = sys.modules.get("rmsnorm_fwd_bwd_03_gb300")
    if mod is None or getattr(mod, "_lib", None) is None or not gpu_available():
        return
    import torch
    torch.cuda.synchronize()
    assert mod.device_error() == 0, "a kernel reported a wait timeout (device error word != 0)"
