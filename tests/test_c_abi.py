"""The C ABI from a plain C11 program (tests/c/thd_roundtrip.c): it compiles
and links against include/thd.h and libthd.so without a GPU, and runs on one."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "thd_roundtrip.c")
PKG = os.path.join(ROOT, "context_packed_sequence_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cuda_lib_dir():
    import glob
    for d in [os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib")] + glob.glob(os.path.join(CUDA, "targets", "*", "lib")):
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    pytest.skip("no libcudart.so under the CUDA toolkit")


def _compile(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(PKG, "libthd.so")):
        from context_packed_sequence_gb300 import build
        build.build()
    exe = str(tmp_path / "thd_roundtrip")
    cmd = [cc, "-std=c11", "-Wall", "-Werror", "-O2", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", PKG, "-lthd", f"-Wl,-rpath,{PKG}",
           "-L", _cuda_lib_dir(), "-lcudart", f"-Wl,-rpath,{_cuda_lib_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


def test_debug_header_links_against_the_checked_build(tmp_path):
    """include/thd_debug.h is plain C too, and its entry points resolve in
    libthd_checked.so (the default library does not export them)."""
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    checked = os.path.join(PKG, "libthd_checked.so")
    if not os.path.exists(checked):
        from context_packed_sequence_gb300 import build
        build.build(checked=True)
    src = tmp_path / "debug.c"
    src.write_text('#include "thd_debug.h"\n'
                   "int main(void) {\n"
                   "  thd_status_t (*a)(cudaStream_t) = thd_debug_stall_next_bulk_copy;\n"
                   "  thd_status_t (*b)(cudaStream_t) = thd_debug_stall_next_ulysses_tile;\n"
                   "  thd_status_t (*c)(cudaStream_t) = thd_debug_stall_next_pack;\n"
                   "  return (a != 0 && b != 0 && c != 0) ? 0 : 1;\n"
                   "}\n")
    exe = str(tmp_path / "debug")
    cmd = [cc, "-std=c11", "-Wall", "-Werror", "-O2", str(src), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", PKG, "-l:libthd_checked.so", f"-Wl,-rpath,{PKG}",
           "-L", _cuda_lib_dir(), "-lcudart", f"-Wl,-rpath,{_cuda_lib_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
