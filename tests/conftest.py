import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--record-errors", default=None,
                     help="write the largest parity error seen per test family to this JSON file")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionfinish(session, exitstatus):
    path = session.config.getoption("--record-errors")
    if path:
        import helpers
        with open(path, "w") as f:
            json.dump({k: {"max": v, "test": helpers.OBSERVED_AT.get(k)} for k, v in helpers.OBSERVED.items()}, f,
                      indent=1, sort_keys=True)


@pytest.fixture(scope="session")
def repo_root():
    return ROOT
