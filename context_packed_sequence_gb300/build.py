"""Build libthd.so in-tree with nvcc for sm_103a (GB300).

Every ``csrc/*.cu`` translation unit is compiled in parallel into
``_build/thd/`` at the repository root, then linked into
``context_packed_sequence_gb300/libthd.so`` (CUDA runtime linked statically,
so the library loads without any library path set up).  ``--checked`` builds
the debug variant ``libthd_checked.so`` (``-DTHD_CHECKED=1``: every computed
row index is range-checked in the kernels), which the package loads when
``THD_CHECKED=1`` is set in the environment.

    python -m context_packed_sequence_gb300.build [--checked]
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "thd")
LIB = os.path.join(PKG, "libthd.so")
BUILD_CHECKED = os.path.join(ROOT, "_build", "thd_checked")
LIB_CHECKED = os.path.join(PKG, "libthd_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libthd")


def sources() -> list:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(args):
    src, obj, extra = args
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, cmd, r


def _variant(checked: bool, extra_flags=()):
    build_dir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    flags = list(extra_flags) + (["-DTHD_CHECKED=1"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    jobs = [(src, os.path.join(build_dir, os.path.basename(src)[:-3] + ".o"), flags) for src in sources()]
    return lib_path, jobs


def _build(variants, verbose: bool = False) -> list:
    """Compile every variant's translation units in one parallel pool, then
    link each library."""
    jobs = [j for _, js in variants for j in js]
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(_compile, jobs))
    failed = False
    for src, cmd, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        failed |= r.returncode != 0
    if failed:
        raise RuntimeError("libthd: compilation failed (see the nvcc output above)")
    for lib_path, js in variants:
        tmp = lib_path + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[j[1] for j in js]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError("libthd: link failed")
        os.replace(tmp, lib_path)
    return [lib_path for lib_path, _ in variants]


def build(extra_flags=(), verbose: bool = False, checked: bool = False) -> str:
    """Build libthd.so (or, with checked, libthd_checked.so)."""
    return _build([_variant(checked, extra_flags)], verbose)[0]


def build_all(extra_flags=(), verbose: bool = False) -> list:
    """Build libthd.so and libthd_checked.so together."""
    return _build([_variant(False, extra_flags), _variant(True, extra_flags)], verbose)


if __name__ == "__main__":
    args = sys.argv[1:]
    print(build(extra_flags=[a for a in args if a != "--checked"], verbose=True, checked="--checked" in args))
