"""The C ABI without a GPU: the library loads, exports every declared symbol,
and its host-side logic (argument checks, quick returns, kernel choice) behaves
as include/sgemm_gb300.h states.  No call here reaches the CUDA runtime."""

import ctypes
import os
import re

import pytest

import dense_fp32_matrix_row_gb300 as sg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def L():
    sg.build()
    return sg.lib()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "sgemm" in names and "sgemm_3xtf32" in names and len(names) >= 9
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10):
        s = sg.status_string(code)
        assert s and s != "unknown status"
    assert sg.status_string(12345) == "unknown status"
    assert sg.version() >= 100


def sel(M, N, K, **kw):
    return sg.select_kernel(M, N, K, **kw)


def test_argument_errors(L):
    assert sel(-1, 4, 4) == sg.ERR_BAD_DIM
    assert sel(4, -1, 4) == sg.ERR_BAD_DIM
    assert sel(4, 4, -1) == sg.ERR_BAD_DIM
    assert sel(4, 4, 4, lda=3) == sg.ERR_BAD_LD
    assert sel(4, 4, 4, ldb=3) == sg.ERR_BAD_LD
    assert sel(4, 4, 4, ldc=3) == sg.ERR_BAD_LD
    assert sel(4, 4, 4, C=0) == sg.ERR_NULL_PTR
    assert sel(4, 4, 4, A=0) == sg.ERR_NULL_PTR
    assert sel(4, 4, 4, B=0) == sg.ERR_NULL_PTR
    # C overlapping A or B (address ranges in bytes)
    assert sel(64, 64, 64, A=1 << 20, C=(1 << 20) + 4 * 100) == sg.ERR_ALIAS
    assert sel(64, 64, 64, B=1 << 20, C=(1 << 20) - 4 * 100) == sg.ERR_ALIAS
    assert sel(64, 64, 64, A=1 << 20, B=1 << 22, C=1 << 24) == sg.KERNEL_FFMA_GENERIC
    # enormous sizes are rejected instead of overflowing offsets
    assert sel(1 << 40, 1 << 20, 4, A=1 << 20, B=1 << 22, C=1 << 24) == sg.ERR_BAD_DIM


def test_quick_returns(L):
    assert sel(0, 5, 5) == sg.KERNEL_NONE
    assert sel(5, 0, 5) == sg.KERNEL_NONE
    assert sel(0, 5, 5, C=0) == sg.KERNEL_NONE            # nothing is touched
    assert sel(5, 5, 0, A=0, B=0) == sg.KERNEL_SCALE_C    # K == 0: A, B unused
    assert sel(5, 5, 5, alpha=0.0, A=0, B=0) == sg.KERNEL_SCALE_C


def test_kernel_choice(L):
    a, b, c = 1 << 20, 1 << 26, 1 << 30
    for M in (1, 4, 16):
        assert sel(M, 14336, 4096, A=a, B=b, C=c) == sg.KERNEL_DECODE
    assert sel(17, 640, 640, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA
    assert sel(4092, 4092, 4092, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA
    # tiny products (at most 2^21 multiply-adds) take the one-launch plain-load kernel
    assert sel(128, 128, 128, A=a, B=b, C=c) == sg.KERNEL_FFMA_GENERIC
    assert sel(17, 64, 64, A=a, B=b, C=c) == sg.KERNEL_FFMA_GENERIC
    assert sel(129, 128, 128, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA
    # B misaligned or ldb % 4 != 0 -> plain-load kernel; A may be anything
    # (the TMA path reads A through its transposed copy)
    assert sel(256, 128, 128, A=a + 4, B=b, C=c) == sg.KERNEL_FFMA_TMA
    assert sel(256, 128, 127, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA       # lda = 127
    assert sel(256, 128, 128, A=a, B=b + 8, C=c) == sg.KERNEL_FFMA_GENERIC
    assert sel(256, 130, 128, A=a, B=b, C=c) == sg.KERNEL_FFMA_GENERIC   # ldb = 130
    # C alignment does not matter for the choice (the epilogue adapts)
    assert sel(256, 128, 128, A=a, B=b, C=c + 4) == sg.KERNEL_FFMA_TMA


def test_tensor_core_modes(L):
    a, b, c = 1 << 20, 1 << 26, 1 << 30
    assert sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=True) == sg.KERNEL_TF32X3
    assert sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=sg.MODE_3XTF32) == sg.KERNEL_TF32X3
    assert sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=sg.MODE_TF32) == sg.KERNEL_TF32
    assert sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=sg.MODE_BF16) == sg.KERNEL_BF16
    # any alignment: both tensor-core paths read rounded / split copies
    assert sel(256, 130, 127, A=a + 4, B=b + 8, C=c, tensor_cores=sg.MODE_TF32) == sg.KERNEL_TF32
    # skinny products stay on the FP32 decode kernel in every mode
    for mode in (sg.MODE_FP32, sg.MODE_3XTF32, sg.MODE_TF32, sg.MODE_BF16):
        assert sel(16, 14336, 4096, A=a, B=b, C=c, tensor_cores=mode) == sg.KERNEL_DECODE
    assert sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=sg.MODE_FP32) == sg.KERNEL_FFMA_TMA
    # an unknown mode is an argument error in the C ABI
    assert L.sgemm_select_kernel(256, 256, 256, 1.0, a, 256, b, 256, 0.0, c, 256, 7) == sg.ERR_BAD_ARG
    with pytest.raises(ValueError):
        sel(256, 256, 256, A=a, B=b, C=c, tensor_cores=5)


def test_force_kernel(L):
    a, b, c = 1 << 20, 1 << 26, 1 << 30
    assert sg.force_kernel(99) == sg.ERR_BAD_ARG
    prev = sg.force_kernel(sg.KERNEL_FFMA_GENERIC)
    try:
        assert prev == sg.KERNEL_AUTO
        assert sel(256, 256, 256, A=a, B=b, C=c) == sg.KERNEL_FFMA_GENERIC
        sg.force_kernel(sg.KERNEL_DECODE)
        assert sel(256, 256, 256, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA   # decode cannot take M > 16
        sg.force_kernel(sg.KERNEL_FFMA_TMA)
        assert sel(8, 256, 256, A=a, B=b, C=c) == sg.KERNEL_FFMA_TMA
        assert sel(8, 256, 256, A=a, B=b + 4, C=c) == sg.KERNEL_DECODE  # TMA cannot take it
    finally:
        sg.force_kernel(sg.KERNEL_AUTO)


def test_rejected_calls_touch_nothing(L):
    # These return before any CUDA call, so they work without a GPU.
    assert sg.sgemm_ptr(-1, 1, 1, 1.0, 16, 1, 16, 1, 0.0, 16, 1) == sg.ERR_BAD_DIM
    assert sg.sgemm_ptr(0, 7, 7, 1.0, None, 7, None, 7, 0.0, None, 7) == sg.OK
    assert sg.sgemm_ptr(3, 3, 3, 1.0, 16, 2, 64, 3, 0.0, 256, 3) == sg.ERR_BAD_LD
    assert sg.sgemm_ptr(3, 3, 3, 1.0, 16, 3, 64, 3, 0.0, 20, 3) == sg.ERR_ALIAS


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(sg, "_lib", None)
    monkeypatch.setattr(sg, "LIBRARY", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        sg.lib()


def host_call(L, M, N, K, A=1 << 20, lda=None, B=1 << 26, ldb=None, C=1 << 32, ldc=None,
              mode=0, alpha=1.0, beta=0.0):
    return int(L.sgemm_host(M, N, K, alpha, A, K if lda is None else lda, B,
                            N if ldb is None else ldb, beta, C, N if ldc is None else ldc, mode,
                            None))


def test_host_path_argument_errors(L):
    # rejected on the host before any CUDA call (none would succeed here)
    assert host_call(L, -1, 4, 4) == sg.ERR_BAD_DIM
    assert host_call(L, 4, 4, 4, lda=3) == sg.ERR_BAD_LD
    assert host_call(L, 4, 4, 4, ldc=3) == sg.ERR_BAD_LD
    assert host_call(L, 4, 4, 4, C=0) == sg.ERR_NULL_PTR
    assert host_call(L, 64, 64, 64, A=1 << 20, C=(1 << 20) + 400) == sg.ERR_ALIAS
    assert host_call(L, 4, 4, 4, mode=9) == sg.ERR_BAD_ARG
    assert host_call(L, 0, 4, 4) == sg.OK   # nothing to do
    assert L.sgemm_host_set_panels(-1) == sg.ERR_BAD_ARG


def test_host_path_panels(L):
    prev = sg.host_set_panels(0)
    try:
        # skinny products and products without A@B: one panel
        assert sg.host_panel_rows(16, 14336, 4096) == 16
        assert sg.host_panel_rows(256, 4096, 4096) == 256
        assert sg.host_panel_rows(5000, 4096, 0) == 5000
        assert sg.host_panel_rows(0, 5, 5) == 0
        assert sg.host_panel_rows(-1, 5, 5) == sg.ERR_BAD_DIM
        for M, N in ((4092, 4092), (8192, 8192), (8192, 14336), (1000, 300), (300, 20000)):
            r = sg.host_panel_rows(M, N, 4096)
            assert 1 <= r <= M
            assert r == M or r % 128 == 0
            assert -(-M // r) <= 8
        # forced counts: rows rounded up to 128, never more panels than asked
        for P in (1, 2, 3, 5, 8):
            sg.host_set_panels(P)
            r = sg.host_panel_rows(4092, 4092, 4092)
            assert r == (4092 if P == 1 else min(4092, -(-(-(-4092 // P)) // 128) * 128))
            assert -(-4092 // r) <= P
        assert sg.host_set_panels(0) == 8
    finally:
        sg.host_set_panels(prev)
