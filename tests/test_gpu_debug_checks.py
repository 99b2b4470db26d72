"""The bounds-checked debug build (libddt_checks.so, compiled with -DDDT_CHECKS).

Its kernels test every computed cache row, page index, TMA coordinate and
output row before the access; a failed check skips or clamps the access,
counts the failure and sets DDT_ST_CHECK in the sequence's status. Here the
unit-walking attention cases, the whole step (sweep points and edge cases),
accept and compaction, and the NEXT rows run against that library in a
child process, with every test also asserting that no check failed (the
autouse fixture in conftest.py); the parity assertions of those tests apply
as well.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["tests/test_gpu_attn_units.py", "tests/test_gpu_step.py",
         "tests/test_gpu_accept_compact.py", "tests/test_gpu_rope_append.py",
         "tests/test_gpu_drafter_topk.py", "tests/test_gpu_target_argmax.py"]


def test_release_library_reports_no_checks(lib):
    from tree_speculative_decoding_ddt_gb300 import _binding
    if os.environ.get("DDT_LIB") == "checks":
        pytest.skip("this process runs the debug build")
    built, n_failed, first = _binding.debug_checks()
    assert (built, n_failed, first) == (False, 0, 0)


def test_suites_pass_on_the_bounds_checked_build():
    if os.environ.get("DDT_LIB") == "checks":
        pytest.skip("already inside the debug-build run")
    lib = os.path.join(ROOT, "tree_speculative_decoding_ddt_gb300", "libddt_checks.so")
    assert os.path.exists(lib), "libddt_checks.so is not built (build() makes both libraries)"
    env = dict(os.environ, DDT_LIB="checks")
    r = subprocess.run([sys.executable, "-m", "pytest", *FILES, "-x", "-q", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-15:])
    assert r.returncode == 0, tail
    assert " passed" in tail
