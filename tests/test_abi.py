"""The C-ABI library loads and exports every entry point include/ddt.h
declares; host-side argument checks answer without any GPU work."""
import ctypes
import os
import re

import pytest

from tree_speculative_decoding_ddt_gb300 import _binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ddt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ddt_[a-z_0-9]+)\s*\(",
                                 src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_ddt_gb300 import build
    build.build()
    return B.load()


def test_header_declares_the_five_calls():
    names = declared_functions()
    for n in ("ddt_tree_build", "ddt_verify_attn", "ddt_tree_accept", "ddt_cache_compact",
              "ddt_step"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in B.SIGNATURES, f"{n} has no binding signature"


def test_strerror_and_version(lib):
    assert lib.ddt_abi_version() == 1
    assert lib.ddt_strerror(0) == b"ok"
    assert lib.ddt_strerror(-1) == b"invalid argument"
    assert b"unknown" in lib.ddt_strerror(-99)


def test_struct_layouts_match_the_header():
    assert ctypes.sizeof(B.TreeDims) == 20
    assert ctypes.sizeof(B.AttnDims) == 48
    assert B.AttnDims.kv_rows.offset == 32 and B.AttnDims.scale.offset == 40


def test_host_side_argument_errors(lib):
    bad = B.TreeDims(0, 4, 4, 8, 100)
    assert lib.ddt_tree_build(ctypes.byref(bad), *([None] * 12), None) == -1
    big = B.TreeDims(1, 4, 4, 200, 100)
    assert lib.ddt_tree_build(ctypes.byref(big), *([None] * 12), None) == -2
    assert lib.ddt_tree_accept(0, 9, 4, *([None] * 9)) == -1
    assert lib.ddt_tree_accept(1, 129, 4, *([None] * 9)) == -2
    assert lib.ddt_cache_compact(1, 4, 1152, 64, 1, 100, None, None, None, None, None, None, None,
                                 None) == -1
    d = B.attn_dims(1, 9, 64, 512, 64, 64, 1, 100, B.DDT_BF16, 0.1, 100)
    assert lib.ddt_verify_attn(ctypes.byref(d), *([None] * 10), 0, None) == -1  # null pointers
    assert lib.ddt_verify_attn(ctypes.byref(d), *([None] * 10), 0, None) == -1
    d = B.attn_dims(1, 9, 64, 256, 64, 64, 1, 100, B.DDT_BF16, 0.1, 100)
    assert lib.ddt_verify_attn_workspace_size(ctypes.byref(d)) == 0  # C=256 unsupported on bf16
    assert lib.ddt_step(None, None) == -1


def test_host_side_errors_of_the_next_rows(lib):
    # no pointer is dereferenced and nothing is launched: every call is
    # refused on the host
    assert lib.ddt_target_argmax(0, 10, B.DDT_BF16, None, None, None) == -1
    assert lib.ddt_drafter_topk(4, 10, 17, B.DDT_BF16, 1, 1, 1, None) == -2
    assert lib.ddt_drafter_topk(4, 10, 11, B.DDT_BF16, 1, 1, 1, None) == -2  # K > V
    dims = B.attn_dims(1, 2, 1, 8, 7, 4, 1, 8, B.DDT_BF16, 1.0, 0)       # odd R
    assert lib.ddt_rope_append(ctypes.byref(dims), 10000.0, *([1] * 8), None) == -1
    dims = B.attn_dims(1, 2, 1, 8, 8, 4, 1, 8, B.DDT_BF16, 1.0, 0)
    assert lib.ddt_rope_append(ctypes.byref(dims), 0.0, *([1] * 8), None) == -1
    assert lib.ddt_rope_append(ctypes.byref(dims), 10000.0, None, *([1] * 7), None) == -1
    a = B.LoopArgs()
    assert lib.ddt_loop_workspace_size(ctypes.byref(a)) == 0
    h = ctypes.c_void_p()
    assert lib.ddt_loop_create(ctypes.byref(a), ctypes.byref(h)) == -1 and not h.value
    assert lib.ddt_loop_launch(None, None) == -1
    assert lib.ddt_loop_destroy(None) == 0
