"""Failure detection on the device: the bounded waits every kernel uses give
up after about a second and report DDT_ST_TIMEOUT instead of hanging, and the
GPU stays usable afterwards (a wait on a phase nothing completes, in a small
kernel of its own; no fault, trap or endless loop is involved)."""
import pytest
import torch

from tree_speculative_decoding_ddt_gb300 import _binding as DB

pytestmark = pytest.mark.gpu


def test_a_wait_nothing_completes_gives_up_after_about_a_second():
    stuck, done, ms = DB.ddt_wait_selftest()
    assert stuck == DB.ST_TIMEOUT
    assert done == 0
    assert 900 <= ms <= 3000
    # the context is still usable
    x = torch.arange(10, device="cuda")
    assert int(x.sum()) == 45
