import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libqmm")


@pytest.fixture(scope="session", autouse=True)
def _build_host_libs():
    """Compile the generator and the oracle (host C) once per session."""
    import oracle
    import synth
    synth.build()
    oracle.build()


@pytest.fixture(params=[1, 2], ids=["mma_sync", "tcgen05"])
def backend(request):
    """Both kernel backends run every GPU parity and invariance test."""
    return request.param
