import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def deterministic_backward():
    """Run the test with the library's deterministic backward (no sums in
    global memory at any head size), then restore the default."""
    import online_softmax_05_gb300 as fa
    from online_softmax_05_gb300 import build
    build.build()
    lib = fa.load_library()
    assert lib.fa_set_deterministic(1) == 0
    try:
        yield
    finally:
        lib.fa_set_deterministic(0)

