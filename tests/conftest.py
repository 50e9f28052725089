import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large CPU or GPU case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree.  GPU tests fail (not skip) without it."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test ran without a CUDA device")
    import matrix_optimizer_step_gb300 as mos

    mos.load_library()
    return mos
