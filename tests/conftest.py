import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def kda_lib():
    """The CUDA library, built in-tree if it is missing or stale."""
    from gated_delta_rule_30_gb300 import build
    build.build()
    import gated_delta_rule_30_gb300 as kda
    kda.lib()
    return kda
