import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libxt.so")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _output_guards(request):
    """After every GPU test: the guard bands around the outputs it allocated are intact."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from tests import gpu_util
    import torch
    torch.cuda.synchronize()
    bad = gpu_util.check_guards()
    assert not bad, "; ".join(bad[:5])
