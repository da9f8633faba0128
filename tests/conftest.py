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
    parser.addoption("--checked-lib", action="store_true",
                     help="run every GPU test through the bounds-checked build (libsptp_check.so): each kernel "
                          "checks the indices and addresses it computes and reports a violation in the status "
                          "words that the tests read")


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


@pytest.fixture(scope="session", autouse=True)
def _checked_library(request):
    """With --checked-lib, the bounds-checked build is the library every test
    loads (the tests' own load_library() calls keep it)."""
    if not request.config.getoption("--checked-lib"):
        yield
        return
    import torch
    if not torch.cuda.is_available():
        yield
        return
    import sequence_tensor_transformer_gb300 as st
    from sequence_tensor_transformer_gb300 import build
    st.load_library(build.build(checked=True), replace=True)
    yield
