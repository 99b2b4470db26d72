"""Builds ``libddt.so`` in-tree for sm_103a with nvcc.

Each ``csrc/*.cu`` file compiles to an object in ``_build/`` (in parallel),
then nvcc links them into ``libddt.so`` next to this file. The CUDA runtime
is linked statically, so the library needs only the NVIDIA driver at run
time. ``build(checks=True)`` makes the debug variant ``libddt_checks.so``
(objects in ``_build_checks/``, compiled with ``-DDDT_CHECKS``: device bounds
checks that record a status instead of faulting).
``python -m tree_speculative_decoding_ddt_gb300.build [--checks]`` runs it.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libddt.so")
BUILD_CHECKS = os.path.join(HERE, "_build_checks")
LIB_CHECKS = os.path.join(HERE, "libddt_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libddt")
    return exe


def _compile(src: str, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(verbose_ptxas: bool = False, force: bool = False, checks: bool = False) -> str:
    """Compile and link; returns the path of ``libddt.so`` (``libddt_checks.so``
    with ``checks``)."""
    build_dir, lib = (BUILD_CHECKS, LIB_CHECKS) if checks else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "ddt.h")]
    newest = max(os.path.getmtime(p) for p in sources + headers + [__file__])
    if not force and not verbose_ptxas and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checks:
        extra = extra + ["-DDDT_CHECKS"]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(sources)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), sources))
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, force=True, checks="--checks" in sys.argv))
