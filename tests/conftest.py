import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    """The CPU oracle module (compiled on first use)."""
    from oracle import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session", autouse=True)
def _guard_bands_installed():
    """With a GPU, every cache array and decode buffer the binding allocates
    sits between guard bands (tests/guard.py)."""
    import torch
    if not torch.cuda.is_available():
        yield
        return
    import guard
    mp = pytest.MonkeyPatch()
    guard.install(mp)
    yield
    mp.undo()


@pytest.fixture(autouse=True)
def _guard_bands_checked(request):
    """After each GPU test: no kvq kernel wrote outside its buffers."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if torch.cuda.is_available():
        import guard
        guard.check_and_release()
