"""sgemm_noalloc: the entry point for callers that must not allocate device memory.

Some users of the library cannot let it call cudaMalloc or cudaMallocAsync:
their device memory is all reserved up front by their own pool or by a host
framework, or the call sits on a latency-critical path.  sgemm_noalloc keeps
the FFMA kernel's transposed copy of A in a fixed array compiled into the
library instead of a workspace it allocates.  These tests call it through the
C ABI and check it against sgemm() -- the entry point that does allocate --
within the parity gate, on two calls in a row (the second call reuses the
array the first one left behind), and check that oversized problems are
refused.  The file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest

import synth
from gpu_util import GATE, normwise_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402

_i64, _f32, _vp = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
SGEMM_ERR_TOO_LARGE = -9


@pytest.fixture(scope="module")
def noalloc():
    sg.build()
    fn = sg.lib().sgemm_noalloc
    fn.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]
    fn.restype = ctypes.c_int
    return fn


def _compare_one(noalloc, M, N, K, alpha, beta, seed):
    A = synth.matrix(M, K, seed=seed, stream=0, dist="normal")
    B = synth.matrix(K, N, seed=seed, stream=1, dist="normal")
    C0 = synth.matrix(M, N, seed=seed, stream=2, dist="normal")
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    want = torch.from_numpy(C0).cuda()
    got = want.clone()
    kid = sg.select_kernel(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                           got.data_ptr(), N)
    assert kid == sg.KERNEL_FFMA_TMA, "these shapes must take the scratch-using kernel"
    stream = torch.cuda.current_stream().cuda_stream
    sg.sgemm(dA, dB, want, alpha, beta)
    rc = noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, got.data_ptr(), N,
                 stream)
    assert rc == sg.OK, sg.status_string(rc)
    assert sg.status() == sg.OK
    err = normwise_err(got.cpu().numpy(), want.cpu().numpy(), A, B, K, alpha, beta, C0)
    assert err <= GATE, f"sgemm_noalloc differs from sgemm: {err:.3e}"


def test_matches_sgemm_on_two_calls_in_a_row(noalloc):
    # The first call fills more of the array than the second reads.
    _compare_one(noalloc, 1000, 700, 1500, 1.0, 0.5, seed=41)
    _compare_one(noalloc, 300, 516, 260, -0.75, 0.0, seed=42)


def test_refuses_problems_beyond_the_array(noalloc):
    # K * round_up(M, 4) = 4100 * 4100 > 16,777,216: refused before any
    # launch, so the (never dereferenced) pointers need only be distinct.
    a, b, c = 1 << 30, 1 << 31, 3 << 30
    M = N = K = 4100
    rc = noalloc(M, N, K, 1.0, a, K, b, N, 0.0, c, N, 0)
    assert rc == SGEMM_ERR_TOO_LARGE
    assert "fixed scratch" in sg.status_string(rc)
    # M = K = 4096 exactly fills the array and is accepted by the size check.
    assert sg.select_kernel(4096, 64, 4096, 1.0, a, 4096, b, 64, 0.0, c, 64) == sg.KERNEL_FFMA_TMA
