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
    # no launch has failed in this thread; names come from the CUDA runtime
    assert lib.ddt_last_cuda_error() == 0
    assert lib.ddt_cuda_error_name(0) == b"cudaSuccess"
    assert lib.ddt_cuda_error_name(1) == b"cudaErrorInvalidValue"


def test_debug_checks_entry_point(lib):
    import ctypes as C
    n, first = C.c_int(7), C.c_int(7)
    # the release library reports no checks and zero counts (no device needed)
    assert lib.ddt_debug_checks(C.byref(n), C.byref(first)) == 0
    assert (n.value, first.value) == (0, 0)
    dbg = os.path.join(os.path.dirname(B.LIB_PATH), "libddt_checks.so")
    if not os.path.exists(dbg):
        pytest.skip("libddt_checks.so not built")
    d = C.CDLL(dbg)
    d.ddt_debug_checks.restype = C.c_int
    d.ddt_debug_checks.argtypes = [C.c_void_p, C.c_void_p]
    assert d.ddt_debug_checks(C.byref(n), C.byref(first)) == 1
    assert n.value == 0


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


def test_struct_layouts_match_a_c_compiler():
    """Every field offset and struct size of the binding's ctypes mirrors
    equals what a C compiler lays out from include/ddt.h."""
    import shutil
    import subprocess
    import tempfile
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("needs a C compiler and the CUDA headers")
    structs = {"ddt_tree_dims": B.TreeDims, "ddt_attn_dims": B.AttnDims,
               "ddt_step_args": B.StepArgs, "ddt_loop_args": B.LoopArgs}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ddt.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for f in py._fields_:
            lines.append(f'  printf("{cname} {f[0]} %zu\\n", offsetof({cname}, {f[0]}));')
    lines += ['  return 0;', '}']
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        open(src, "w").write("\n".join(lines) + "\n")
        subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, src, "-o", exe],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            cname, field, val = line.split()
            got[(cname, field)] = int(val)
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f in py._fields_:
            assert got[(cname, f[0])] == getattr(py, f[0]).offset, (cname, f[0])


def test_loop_arguments_are_checked_on_the_host(lib):
    # each case breaks one rule of ddt_loop_args; nothing reaches the GPU
    def args(**kw):
        a = B.LoopArgs()
        a.tree = B.TreeDims(2, 4, 3, 8, 512)
        a.attn = B.attn_dims(2, 9, 2, 16, 8, 64, 1, 256, B.DDT_F32, 0.25, 128)
        a.theta, a.n_new, a.max_steps, a.golden_len = 10000.0, 12, 64, 20
        for name, _ in B.LoopArgs._fields_[6:-1]:
            setattr(a, name, 64)  # non-null, never dereferenced
        for k, v in kw.items():
            if k in ("B", "D", "K", "budget", "V"):
                setattr(a.tree, k, v)
            elif k in ("Q", "dtype"):
                setattr(a.attn, k, v)
            else:
                setattr(a, k, v)
        return a
    assert lib.ddt_loop_workspace_size(ctypes.byref(args())) > 0
    for bad in (dict(Q=10), dict(B=3), dict(D=0), dict(V=1), dict(n_new=-1),
                dict(max_steps=0), dict(golden_len=1), dict(dtype=7), dict(golden=None),
                dict(accepted=None)):
        a = args(**bad)
        assert lib.ddt_loop_workspace_size(ctypes.byref(a)) == 0, bad
        h = ctypes.c_void_p()
        assert lib.ddt_loop_create(ctypes.byref(a), ctypes.byref(h)) == -1, bad
        assert not h.value
    # valid arguments without a workspace are refused before any capture
    h = ctypes.c_void_p()
    assert lib.ddt_loop_create(ctypes.byref(args(workspace=None)), ctypes.byref(h)) == -4
    assert not h.value


def _cpu(shape, dtype=None):
    import torch
    return torch.zeros(shape, dtype=dtype or torch.bfloat16)


@pytest.mark.parametrize("fn", ["ddt_verify_attn", "ddt_verify_attn_noalloc"])
@pytest.mark.parametrize("kv_shape", [(256, 512), (256, 640), (4, 64, 576), (256,)])
def test_attention_wrappers_refuse_a_malformed_cache_before_any_call(fn, kv_shape):
    # The library views the cache as kv_rows rows of C+R elements; a cache of
    # another shape would be read past its end, so the wrappers refuse it on
    # the shapes alone (these CPU tensors never reach the library).
    import torch
    nb, Q, H, C, R = 1, 9, 4, 512, 64
    args = (_cpu((nb, Q, H, C)), _cpu((nb, Q, H, R)), _cpu(kv_shape),
            _cpu((nb, 4), torch.int32), _cpu((nb,), torch.int32), _cpu((nb, Q, 1), torch.int64))
    with pytest.raises(ValueError, match="kv_cache"):
        getattr(B, fn)(*args, 0.05, 64, 40)


@pytest.mark.parametrize("fn", ["ddt_verify_attn", "ddt_verify_attn_noalloc"])
def test_attention_wrappers_refuse_mismatched_tables(fn):
    import torch
    nb, Q, H, C, R = 2, 9, 4, 512, 64
    good = dict(q_lat=_cpu((nb, Q, H, C)), q_pe=_cpu((nb, Q, H, R)), kv=_cpu((256, C + R)),
                bt=_cpu((nb, 4), torch.int32), pl=_cpu((nb,), torch.int32),
                vis=_cpu((nb, Q, 1), torch.int64))
    for key, bad, what in (("bt", _cpu((1, 4), torch.int32), "block_table"),
                           ("pl", _cpu((3,), torch.int32), "prefix_len"),
                           ("vis", _cpu((nb, Q, 2), torch.int64), "vis_bits"),
                           ("q_pe", _cpu((nb, Q, H + 1, R)), "q_pe")):
        a = dict(good, **{key: bad})
        with pytest.raises(ValueError, match=what):
            getattr(B, fn)(a["q_lat"], a["q_pe"], a["kv"], a["bt"], a["pl"], a["vis"],
                            0.05, 64, 40)
    # well-shaped CPU tensors get past the shape checks and stop at the device check
    with pytest.raises(TypeError, match="CUDA"):
        getattr(B, fn)(*good.values(), 0.05, 64, 40)

