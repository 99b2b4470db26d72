import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The loaded C-ABI library (built in-tree by the package's build step)."""
    from tree_speculative_decoding_ddt_gb300 import _binding
    return _binding.load()


@pytest.fixture(params=["128", "256"])
def attn_rows(request, monkeypatch):
    """Row-tile height of the bf16 verify attention: every case using this
    fixture runs on both kernels (two-CTA 128-row tiles and four-CTA 256-row
    tiles on paired SMs), forced through DDT_VERIFY_ATTN_ROWS."""
    monkeypatch.setenv("DDT_VERIFY_ATTN_ROWS", request.param)
    return int(request.param)


@pytest.fixture(autouse=True)
def _no_failed_bounds_checks(request):
    """Under DDT_LIB=checks (the library built with device bounds checks),
    every GPU test also asserts that no check failed during it."""
    yield
    if os.environ.get("DDT_LIB") != "checks" or request.node.get_closest_marker("gpu") is None:
        return
    import torch
    from tree_speculative_decoding_ddt_gb300 import _binding
    torch.cuda.synchronize()
    built, n_failed, first = _binding.debug_checks()
    assert built, "DDT_LIB=checks but the loaded library was built without DDT_CHECKS"
    assert n_failed == 0, f"{n_failed} device bounds checks failed (first at site {first})"
