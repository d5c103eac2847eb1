"""The debug build: libthd_checked.so (compiled with THD_CHECKED=1, loaded when
THD_CHECKED=1 is set) range-checks every row index its kernels compute in
closed form and reports a miss as THD_ERR_INDEX_RANGE instead of touching
memory.  On the CPU: it builds and exports the same C ABI.  On the GPU: the
parity (including the per-rank copies, the batched swap, packing without
allocation and the single-pass packing), error and maximum-size suites pass against it unchanged, so no
computed index of any of those cases leaves its range."""

import ctypes
import os
import subprocess
import sys

import pytest

from context_packed_sequence_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _checked_env():
    env = dict(os.environ)
    env["THD_CHECKED"] = "1"
    return env


@pytest.fixture(scope="module")
def checked_lib():
    if not os.path.exists(L.CHECKED_LIB_PATH):
        from context_packed_sequence_gb300 import build
        build.build(checked=True)
    return L.CHECKED_LIB_PATH


def test_checked_build_exports_the_abi(checked_lib):
    lib = ctypes.CDLL(checked_lib)
    for name in L.SIGNATURES:
        assert hasattr(lib, name), name
    r = subprocess.run([sys.executable, "-c", "from context_packed_sequence_gb300 import _lib as L; "
                        "L.load(); print(L.lib_path())"], cwd=ROOT, env=_checked_env(), capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == L.CHECKED_LIB_PATH


@pytest.mark.gpu
def test_gpu_suites_pass_on_the_checked_build(checked_lib):
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_parity.py", "tests/test_rank_and_batched.py", "tests/test_errors.py", "tests/test_max_size.py",
           "tests/test_zz_no_alloc.py", "tests/test_pack_onepass.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=_checked_env(), capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
