import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def wan():
    """The CUDA library through its Python binding (built in-tree by __graft_entry__.build())."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from video_vae_decoder_gb300 import binding
    return binding
