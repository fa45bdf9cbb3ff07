"""fp64 CPU oracle for the row-major SGEMM -- TEST INFRASTRUCTURE ONLY.

The C source ``sgemm_oracle.c`` holds the definition (see its header).  This
module compiles it with the host C compiler into ``oracle/_build`` and wraps it
with ctypes for numpy float32 arrays.  Only the tests, the package smoke check
and the benchmark's CPU-baseline leg use it; the CUDA library never does.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "sgemm_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "liboracle_sgemm.so")

# activation ids of oracle_sgemm_rows_fused
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}

_lock = threading.Lock()
_default = None


def compile_library(source: str = SOURCE, output: str = LIBRARY, cc: str | None = None) -> str:
    """Compile an oracle source file into a shared library; returns its path."""
    cc = cc or os.environ.get("CC", "gcc")
    os.makedirs(os.path.dirname(output), exist_ok=True)
    tmp = output + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, output)
    return output


def build() -> str:
    """(Re)build the oracle library if the source is newer than the library."""
    with _lock:
        if (not os.path.exists(LIBRARY)
                or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
            compile_library()
    return LIBRARY


_f32p = ctypes.POINTER(ctypes.c_float)
_i64p = ctypes.POINTER(ctypes.c_int64)


def _ld(x: np.ndarray | None) -> int:
    """Row stride (leading dimension) in elements of a 2-D float32 view."""
    if x is None:
        return 0
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError("oracle operands are 2-D float32 arrays")
    if x.size == 0:
        return max(x.shape[1], 1)
    if x.shape[1] > 1 and x.strides[1] != 4:
        raise ValueError("columns must be contiguous")
    if x.shape[0] <= 1:
        return max(x.shape[1], 1)
    return x.strides[0] // 4


def _ptr(x: np.ndarray | None):
    if x is None:
        return None
    return x.ctypes.data_as(_f32p)


class Oracle:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        self.lib.oracle_sgemm_rows.restype = ctypes.c_int
        self.lib.oracle_sgemm_rows.argtypes = [
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
            _f32p, ctypes.c_int64, _f32p, ctypes.c_int64,
            ctypes.c_float, _f32p, ctypes.c_int64,
            _i64p, ctypes.c_int64, _f32p, ctypes.c_int64, ctypes.c_int]
        self.lib.oracle_sgemm_rows_fused.restype = ctypes.c_int
        self.lib.oracle_sgemm_rows_fused.argtypes = [
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
            _f32p, ctypes.c_int64, _f32p, ctypes.c_int64,
            ctypes.c_float, _f32p, ctypes.c_int64, _f32p, ctypes.c_int,
            _i64p, ctypes.c_int64, _f32p, ctypes.c_int64, ctypes.c_int]
        self.lib.oracle_max_threads.restype = ctypes.c_int
        self.lib.oracle_max_threads.argtypes = []
        self.lib.oracle_round_tf32.restype = None
        self.lib.oracle_round_tf32.argtypes = [_f32p, _f32p, ctypes.c_int64]
        self.lib.oracle_round_bf16.restype = None
        self.lib.oracle_round_bf16.argtypes = [_f32p, _f32p, ctypes.c_int64]

    def round_tf32(self, x: np.ndarray) -> np.ndarray:
        """x rounded to TF32 (nearest, ties away from zero) as a new float32 array."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty_like(x)
        self.lib.oracle_round_tf32(_ptr(x.reshape(-1)), _ptr(out.reshape(-1)), x.size)
        return out

    def round_bf16(self, x: np.ndarray) -> np.ndarray:
        """x rounded to BF16 (nearest, ties to even) as a new float32 array."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty_like(x)
        self.lib.oracle_round_bf16(_ptr(x.reshape(-1)), _ptr(out.reshape(-1)), x.size)
        return out

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def sgemm(self, A: np.ndarray, B: np.ndarray, C0: np.ndarray | None = None,
              alpha: float = 1.0, beta: float = 0.0, rows=None,
              threads: int = 0, bias: np.ndarray | None = None, act: str = "none") -> np.ndarray:
        """act(alpha*A@B + beta*C0 + bias) (rows ``rows`` only, if given) as a new
        float32 array; without ``bias`` and ``act`` the plain product.

        ``A`` is M x K, ``B`` K x N, ``C0`` M x N (may be None when beta == 0),
        ``bias`` N floats added to every row, ``act`` one of ACTIVATIONS.
        Row-strided views (leading dimension > row length) are passed through
        with their strides, so gap columns are never copied or read.
        """
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
        if C0 is not None and C0.shape != (M, N):
            raise ValueError("C0 must be M x N")
        if rows is None:
            rows = np.arange(M, dtype=np.int64)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.empty((rows.size, N), dtype=np.float32)
        if bias is None and act == "none":
            rc = self.lib.oracle_sgemm_rows(
                M, N, K, float(alpha), _ptr(A), _ld(A), _ptr(B), _ld(B),
                float(beta), _ptr(C0), _ld(C0),
                rows.ctypes.data_as(_i64p), rows.size, _ptr(out), max(N, 1), int(threads))
        else:
            if bias is not None:
                bias = np.ascontiguousarray(bias, dtype=np.float32).reshape(-1)
                if bias.size != N:
                    raise ValueError("bias must hold N floats")
            rc = self.lib.oracle_sgemm_rows_fused(
                M, N, K, float(alpha), _ptr(A), _ld(A), _ptr(B), _ld(B),
                float(beta), _ptr(C0), _ld(C0), _ptr(bias), ACTIVATIONS[act],
                rows.ctypes.data_as(_i64p), rows.size, _ptr(out), max(N, 1), int(threads))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return out


def default() -> Oracle:
    """The oracle built from ``sgemm_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        try:
            _default = Oracle(build())
        except OSError:   # a library built for another machine: rebuild it here
            with _lock:
                compile_library()
            _default = Oracle(LIBRARY)
    return _default


def sgemm(A, B, C0=None, alpha=1.0, beta=0.0, rows=None, threads=0, inputs="fp32",
          bias=None, act="none"):
    """act(alpha*A@B + beta*C0 + bias) from the default oracle build (see
    ``Oracle.sgemm``).

    ``inputs="tf32"`` / ``"bf16"`` give the reduced-precision products: A and B
    are rounded to TF32 / BF16 first (``round_tf32`` / ``round_bf16``), C0 and
    bias are not."""
    if inputs == "tf32":
        A, B = round_tf32(A), round_tf32(B)
    elif inputs == "bf16":
        A, B = round_bf16(A), round_bf16(B)
    elif inputs != "fp32":
        raise ValueError(f"unknown input precision {inputs!r}")
    return default().sgemm(A, B, C0, alpha=alpha, beta=beta, rows=rows, threads=threads,
                           bias=bias, act=act)


def round_tf32(x):
    """x rounded to TF32, nearest with ties away from zero (see ``oracle_round_tf32``)."""
    return default().round_tf32(x)


def round_bf16(x):
    """x rounded to BF16, nearest with ties to even (see ``oracle_round_bf16``)."""
    return default().round_bf16(x)
