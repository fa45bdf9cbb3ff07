"""Row-major FP32 GEMM for GB300 (sm_103a): Python binding of ``libsgemm_gb300.so``.

``C <- alpha * A @ B + beta * C`` with A M x K, B K x N, C M x N, row-major
(the operation of "GPU GEMM 优化完全拆解（一）", section "什么是 GEMM").  Every
step runs in the library's CUDA kernels; this module only marshals arguments
(torch CUDA tensors or raw device pointers) into the C ABI declared in
``include/sgemm_gb300.h``.  There is no CPU path: if the library is missing,
calls raise.
"""

from __future__ import annotations

import ctypes
import os

from .build import LIBRARY, build  # noqa: F401  (build is part of the public API)

__all__ = ["sgemm", "sgemm_host", "host_set_panels", "host_panel_rows", "sgemm_3xtf32", "sgemm_tf32", "sgemm_bf16", "sgemm_ptr", "status", "select_kernel",
           "force_kernel", "ffma_configs", "ffma_config_for", "ffma_force_config", "ffma_force_tail_sum", "ffma_tail_plan", "kernel_timing", "kernel_timing_result", "set_wait_limit", "selftest_wait", "release_workspaces", "status_string",
           "version", "SgemmError", "lib"]

OK = 0
ERR_BAD_DIM, ERR_BAD_LD, ERR_NULL_PTR, ERR_ALIAS = -1, -2, -3, -4
ERR_CUDA, ERR_DEVICE, ERR_TIMEOUT, ERR_BAD_ARG = -5, -6, -7, -8
ERR_TOO_LARGE, ERR_CAPTURE = -9, -10

KERNEL_AUTO, KERNEL_NONE, KERNEL_SCALE_C, KERNEL_FFMA_TMA = 0, 1, 2, 3
KERNEL_FFMA_GENERIC, KERNEL_DECODE, KERNEL_TF32X3, KERNEL_TF32, KERNEL_BF16 = 4, 5, 6, 7, 8
KERNEL_NAMES = {KERNEL_NONE: "none", KERNEL_SCALE_C: "scale_c", KERNEL_FFMA_TMA: "ffma_tma",
                KERNEL_FFMA_GENERIC: "ffma_generic", KERNEL_DECODE: "decode",
                KERNEL_TF32X3: "tf32x3", KERNEL_TF32: "tf32", KERNEL_BF16: "bf16"}
# activations of the fused epilogue (sgemm_fused)
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}
# arithmetic of a call (sgemm, sgemm_3xtf32, sgemm_tf32)
MODE_FP32, MODE_3XTF32, MODE_TF32, MODE_BF16 = 0, 1, 2, 3
_ENTRY = {MODE_FP32: "sgemm", MODE_3XTF32: "sgemm_3xtf32", MODE_TF32: "sgemm_tf32",
          MODE_BF16: "sgemm_bf16"}


def _mode(tensor_cores) -> int:
    """False/True (FP32 / 3xTF32) or one of the MODE_* values."""
    if tensor_cores is True:
        return MODE_3XTF32
    if tensor_cores is False or tensor_cores is None:
        return MODE_FP32
    if tensor_cores in _ENTRY:
        return int(tensor_cores)
    raise ValueError(f"unknown arithmetic mode {tensor_cores!r}")


class SgemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else
                         f"{status_string(code)} ({code})")


_lib = None
_i64, _f32, _vp = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_GEMM_ARGS = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIBRARY):
            raise RuntimeError(
                f"CUDA library {LIBRARY} is not built; run "
                "`python -m dense_fp32_matrix_row_gb300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(LIBRARY)
        for name in ("sgemm", "sgemm_3xtf32", "sgemm_tf32", "sgemm_bf16"):
            getattr(L, name).argtypes = _GEMM_ARGS
            getattr(L, name).restype = ctypes.c_int
        L.sgemm_fused.argtypes = _GEMM_ARGS[:-1] + [_vp, ctypes.c_int, ctypes.c_int, _vp]
        L.sgemm_fused.restype = ctypes.c_int
        L.sgemm_host.argtypes = _GEMM_ARGS[:-1] + [ctypes.c_int, _vp]
        L.sgemm_host.restype = ctypes.c_int
        L.sgemm_host_set_panels.argtypes = [ctypes.c_int]
        L.sgemm_host_set_panels.restype = ctypes.c_int
        L.sgemm_host_panel_rows.argtypes = [_i64, _i64, _i64]
        L.sgemm_host_panel_rows.restype = _i64
        L.sgemm_select_kernel.argtypes = _GEMM_ARGS[:-1] + [ctypes.c_int]
        L.sgemm_ffma_config_for.argtypes = [_i64, _i64, _i64]
        L.sgemm_ffma_config_for.restype = ctypes.c_int
        L.sgemm_select_kernel.restype = ctypes.c_int
        L.sgemm_status.argtypes = [_vp]
        L.sgemm_status.restype = ctypes.c_int
        L.sgemm_status_string.argtypes = [ctypes.c_int]
        L.sgemm_status_string.restype = ctypes.c_char_p
        L.sgemm_force_kernel.argtypes = [ctypes.c_int]
        L.sgemm_force_kernel.restype = ctypes.c_int
        L.sgemm_set_wait_limit.argtypes = [_i64]
        L.sgemm_set_wait_limit.restype = _i64
        L.sgemm_selftest_wait.argtypes = [_i64, _vp]
        L.sgemm_selftest_wait.restype = ctypes.c_int
        L.sgemm_release_workspaces.argtypes = []
        L.sgemm_release_workspaces.restype = ctypes.c_int
        L.sgemm_version.argtypes = []
        L.sgemm_version.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().sgemm_status_string(int(code)).decode()


def version() -> int:
    return int(lib().sgemm_version())


def _stream_handle(stream, device=None) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream   # torch.cuda.Stream


def _ld(t) -> int:
    """Row stride of a 2-D row-major tensor view (contiguous columns required)."""
    rows, cols = t.shape
    if t.numel() == 0:
        return max(cols, 1)
    if rows == 1:   # the row stride of a single row is arbitrary in torch
        return max(t.stride(0), cols)
    return t.stride(0)


def _check_operand(t, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D float32 tensor")
    if t.numel() and not t.is_cuda:
        raise TypeError(f"{name} must live on a CUDA device")
    if t.shape[1] > 1 and t.stride(1) != 1 and t.numel():
        raise ValueError(f"{name} must be row-major with contiguous rows (stride(1) == 1)")


def sgemm_ptr(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0, tensor_cores=False) -> int:
    """Raw C-ABI call on device pointers; returns the status code.
    ``tensor_cores``: False (sgemm), True (sgemm_3xtf32) or a MODE_* value."""
    fn = getattr(lib(), _ENTRY[_mode(tensor_cores)])
    return int(fn(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream))


def sgemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None,
          tensor_cores: bool = False, bias=None, activation: str = "none") -> None:
    """C <- alpha * A @ B + beta * C in place on torch CUDA float32 tensors.

    A is (M, K), B (K, N), C (M, N); each may be a row-strided view (row
    stride >= row length).  Enqueued on ``stream`` (default: the current torch
    stream of C's device); returns without waiting.  ``tensor_cores`` selects
    the arithmetic: False (FP32 FFMA), True (3xTF32 tcgen05 path) or a MODE_*
    value (MODE_TF32: the reduced-precision 1xTF32 path).  ``bias`` (a CUDA
    float32 tensor of N elements) and ``activation`` (a key of ACTIVATIONS)
    select the fused epilogue C = act(alpha*A@B + beta*C + bias) of
    sgemm_fused.  Raises SgemmError on a rejected call.
    """
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        _check_operand(t, n)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    dev = C.device if C.is_cuda else None
    if bias is None and activation == "none":
        rc = sgemm_ptr(M, N, K, float(alpha), A.data_ptr() or None, _ld(A), B.data_ptr() or None,
                       _ld(B), float(beta), C.data_ptr() or None, _ld(C),
                       _stream_handle(stream, dev), tensor_cores)
        if rc != OK:
            raise SgemmError(rc, _ENTRY[_mode(tensor_cores)])
        return
    if activation not in ACTIVATIONS:
        raise ValueError(f"unknown activation {activation!r}; one of {sorted(ACTIVATIONS)}")
    if bias is not None:
        import torch
        if (not isinstance(bias, torch.Tensor) or bias.dtype != torch.float32 or bias.numel() != N
                or (N and (not bias.is_cuda or not bias.is_contiguous()))):
            raise TypeError("bias must be a contiguous CUDA float32 tensor of N elements")
    rc = int(lib().sgemm_fused(M, N, K, float(alpha), A.data_ptr() or None, _ld(A),
                               B.data_ptr() or None, _ld(B), float(beta), C.data_ptr() or None,
                               _ld(C), bias.data_ptr() if bias is not None and N else None,
                               ACTIVATIONS[activation], _mode(tensor_cores),
                               _stream_handle(stream, dev)))
    if rc != OK:
        raise SgemmError(rc, "sgemm_fused")


def sgemm_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None,
               tensor_cores=False) -> None:
    """C <- alpha * A @ B + beta * C on torch CPU float32 tensors (pinned
    memory lets the copies overlap the compute), through the C ABI's
    sgemm_host: the library copies B and row panels of A and C to the device,
    multiplies each panel as it arrives and copies its rows of C back.
    Enqueued on ``stream`` (default: the current torch stream); C holds the
    result once that stream is synchronised.  ``tensor_cores`` selects the
    arithmetic as in ``sgemm``.  Raises SgemmError on a rejected call."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 2:
            raise TypeError(f"{n} must be a 2-D float32 tensor")
        if t.is_cuda:
            raise TypeError(f"{n} must live in host memory (use sgemm for device tensors)")
        if t.shape[1] > 1 and t.stride(1) != 1 and t.numel():
            raise ValueError(f"{n} must be row-major with contiguous rows (stride(1) == 1)")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, C {tuple(C.shape)}")
    rc = int(lib().sgemm_host(M, N, K, float(alpha), A.data_ptr() or None, _ld(A),
                              B.data_ptr() or None, _ld(B), float(beta), C.data_ptr() or None,
                              _ld(C), _mode(tensor_cores), _stream_handle(stream)))
    if rc != OK:
        raise SgemmError(rc, "sgemm_host")


def host_set_panels(panels: int) -> int:
    """Force sgemm_host's panel count (0: the library's choice); returns the previous setting."""
    rc = int(lib().sgemm_host_set_panels(int(panels)))
    if rc < 0:
        raise SgemmError(rc, "sgemm_host_set_panels")
    return rc


def host_panel_rows(M: int, N: int, K: int) -> int:
    """Rows per panel that sgemm_host would use for this shape."""
    return int(lib().sgemm_host_panel_rows(M, N, K))


def sgemm_3xtf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """``sgemm`` on the 3xTF32 tensor-core path."""
    sgemm(A, B, C, alpha, beta, stream, tensor_cores=True)


def sgemm_tf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """``sgemm`` on the reduced-precision 1xTF32 tensor-core path: A and B are
    rounded to TF32 first (see include/sgemm_gb300.h for the contract)."""
    sgemm(A, B, C, alpha, beta, stream, tensor_cores=MODE_TF32)


def sgemm_bf16(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None) -> None:
    """``sgemm`` on the reduced-precision BF16 tensor-core path: A and B are
    rounded to BF16 first (see include/sgemm_gb300.h for the contract)."""
    sgemm(A, B, C, alpha, beta, stream, tensor_cores=MODE_BF16)


def status(stream=None) -> int:
    """Wait for ``stream`` and return (and clear) the device's kernel error status."""
    return int(lib().sgemm_status(_stream_handle(stream)))


def select_kernel(M, N, K, alpha=1.0, A=16, lda=None, B=16, ldb=None, beta=0.0, C=16, ldc=None,
                  tensor_cores=False) -> int:
    """Kernel id sgemm() would run (host-only).  Pointers may be plain integers."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return int(lib().sgemm_select_kernel(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                         _mode(tensor_cores)))


def force_kernel(kernel_id: int) -> int:
    return int(lib().sgemm_force_kernel(kernel_id))


def ffma_configs() -> list[dict]:
    """The FFMA kernel's compiled tile configurations (index = position)."""
    out = []
    for i in range(int(lib().sgemm_ffma_config_count())):
        v = [ctypes.c_int() for _ in range(6)]
        if lib().sgemm_ffma_config_info(i, *[ctypes.byref(x) for x in v]) != OK:
            raise SgemmError(ERR_BAD_ARG, "sgemm_ffma_config_info")
        out.append(dict(zip(("bm", "bn", "bk", "stages", "threads", "ctas_per_sm"),
                            (x.value for x in v))))
    return out


def ffma_config_for(M: int, N: int, K: int) -> int:
    """The tile configuration an FFMA-path call of this shape runs."""
    return int(lib().sgemm_ffma_config_for(int(M), int(N), int(K)))


def ffma_force_config(idx: int) -> int:
    """Force FFMA tile configuration ``idx`` (-1: the tuning table); returns the previous."""
    return int(lib().sgemm_ffma_force_config(int(idx)))


def ffma_force_tail_sum(mode: int) -> int:
    """How a divided tail's partial tiles are summed (-1 the library's rule,
    0 by the last unit to reach each tile, 1 by a separate kernel); returns
    the previous setting."""
    return int(lib().sgemm_ffma_force_tail_sum(int(mode)))


def ffma_tail_plan(M: int, N: int, K: int) -> dict:
    """The work list an FFMA-path sgemm() call of this shape runs on the
    current device: units (CTAs), span (k-tiles per unit of the divided tail,
    0 if not divided) and tail_sum (1: a separate kernel sums the tail)."""
    units, span, ts = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int()
    f = lib().sgemm_ffma_tail_plan
    f.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 3
    rc = f(int(M), int(N), int(K), ctypes.addressof(units), ctypes.addressof(span), ctypes.addressof(ts))
    if rc != OK:
        raise SgemmError(rc, "sgemm_ffma_tail_plan")
    return {"units": units.value, "span": span.value, "tail_sum": ts.value}


def kernel_timing(enable: bool) -> int:
    """Start (clearing earlier records) or stop bracketing each FFMA tile
    kernel with CUDA events; returns the previous state."""
    rc = int(lib().sgemm_kernel_timing(1 if enable else 0))
    if rc < 0:
        raise SgemmError(rc, "sgemm_kernel_timing")
    return rc


def kernel_timing_result() -> tuple[float, int]:
    """(summed ms, launches) of the FFMA tile kernels recorded since timing started."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    f = lib().sgemm_kernel_timing_result
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    rc = f(ctypes.addressof(ms), ctypes.addressof(n))
    if rc != OK:
        raise SgemmError(rc, "sgemm_kernel_timing_result")
    return ms.value, n.value


def set_wait_limit(ns: int) -> int:
    return int(lib().sgemm_set_wait_limit(int(ns)))


def release_workspaces() -> int:
    """Free the library's cached device workspaces (waits for their streams)."""
    return int(lib().sgemm_release_workspaces())


def selftest_wait(ns: int, stream=None) -> int:
    return int(lib().sgemm_selftest_wait(int(ns), _stream_handle(stream)))
