import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def mla():
    """The library's Python binding, with libmla.so built for sm_103a."""
    import mla_absorbed_latent_02_gb300 as m
    m.build()
    m.load_library()
    return m


@pytest.fixture(scope="session")
def ctx(mla):
    c = mla.Context(0, max_pos=131072)
    yield c
    c.close()
