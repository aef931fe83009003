import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the libvh kernels)")


@pytest.fixture(scope="session")
def orc():
    """The fp64 oracle, built on first use."""
    import oracle
    oracle.build()
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def vhlib():
    """libvh.so, built (for sm_103a) on first use."""
    from visual_backbone_gb300 import _build
    _build.build()
    import visual_backbone_gb300 as vh
    vh.lib()
    return vh
