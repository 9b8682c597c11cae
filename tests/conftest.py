import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the library's kernels)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def orc():
    """The CPU oracle (built on first use)."""
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="module", autouse=True)
def _no_device_faults_after_gpu_module(request):
    """After every GPU test module: the library's device fault word is 0 (no
    kernel gave up on a bounded wait).  Read and cleared, so a fault is charged
    to the module that raised it."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import mxfp4_dequant_matmul_gb300 as mx
    if mx._lib is None:
        return
    faults = mx.mxfp4_device_faults(reset=True)
    assert faults == 0, f"device fault word {faults:#x} after {request.node.name}"
