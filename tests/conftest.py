"""Test configuration: the ``gpu`` marker and session-level builds.

``-m "not gpu"`` runs the oracle pins, the host logic of the library and the
ABI export check on a machine without a GPU; ``-m gpu`` runs the parity tests
that call the CUDA path through the C ABI.
"""
import os
import sys

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if REPO not in sys.path:
    sys.path.insert(0, REPO)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build_oracle()
    return oracle.load()
