import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _clear_device_error(request):
    """Each GPU test starts with a clear device error word (a failed test may leave one set)."""
    if request.node.get_closest_marker("gpu") is not None:
        import torch

        if torch.cuda.is_available():
            from speculative_decoding_attention_gb300 import build as wm_build
            from speculative_decoding_attention_gb300 import wm

            wm_build.build()
            wm.get_device_error()
    yield
