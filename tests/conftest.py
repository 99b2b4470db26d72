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
