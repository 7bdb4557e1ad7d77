import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of CPU or GPU time")


@pytest.fixture(scope="session")
def gpu_lib():
    """The built CUDA library, loaded through its Python binding.

    Fails (does not skip) when a GPU is present but the library is missing:
    there is no CPU fallback to hide behind.
    """
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import distance_argmin_gb300 as km
    km.load()
    return km
