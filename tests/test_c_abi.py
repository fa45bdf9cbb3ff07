"""The C ABI used from plain C: tests/c/sgemm_from_c.c includes only
include/sgemm_gb300.h and the CUDA runtime's C header, allocates device
memory with the CUDA runtime, calls sgemm() and sgemm_host() on small-integer
inputs (exact in FP32, so the result is compared bit for bit with a
double-precision loop) and checks the argument errors.

On CPU the program and the public header are only compiled (as C99, and the
header also as C++); on a GPU the program is built against the in-tree
library and run.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "sgemm_from_c.c")
HEADER = os.path.join(ROOT, "include", "sgemm_gb300.h")


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime.h")):
            return os.path.join(d, "include")
    pytest.skip("CUDA headers not found")


def test_header_is_plain_c_and_cpp():
    cc = shutil.which("gcc") or pytest.skip("no C compiler")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                    "-x", "c", HEADER], check=True)
    cxx = shutil.which("g++") or pytest.skip("no C++ compiler")
    subprocess.run([cxx, "-std=c++11", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", HEADER],
                   check=True)


def test_c_program_compiles():
    cc = shutil.which("gcc") or pytest.skip("no C compiler")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), "-I", _cuda_include(), SRC], check=True)


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_fp32_matrix_row_gb300 as sg
    lib = sg.build()
    from dense_fp32_matrix_row_gb300.build import nvcc
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "sgemm_from_c")
    subprocess.run([nvcc(), SRC, "-I", os.path.join(ROOT, "include"), "-L", libdir,
                    "-lsgemm_gb300", "-Xlinker", "-rpath", "-Xlinker", libdir, "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "sgemm from C: ok" in r.stdout
