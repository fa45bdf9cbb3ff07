"""sgemm_noalloc: the entry point for callers that must not allocate device memory.

Some users of the library cannot let it call cudaMalloc or cudaMallocAsync:
their device memory is all reserved up front by their own pool or by a host
framework, or the call sits on a latency-critical path.  sgemm_noalloc keeps
the FFMA kernel's transposed copy of A in a fixed array compiled into the
library instead of a workspace it allocates.  These tests call it through the
C ABI and check:

  - its output against the fp64 oracle (the parity gate) and against sgemm(),
    the entry point that does allocate, on two calls in a row (the second
    call reuses the array the first one left behind);
  - a problem that fills the array exactly and whose tiles fill less than
    one wave: there is no room for the partial tiles of a divided tail, so the
    tiles run whole (a different summation order from sgemm()'s) and still
    meet the gate;
  - that a call allocates nothing: with every sgemm() workspace released,
    device free memory does not drop across a call, while the same call
    through sgemm() then takes memory for its workspace;
  - that a tensor-core kernel forced with the test hook is refused, and that
    problems beyond the array are refused before any launch.

The file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_util import GATE, normwise_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402

_i64, _f32, _vp = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
SGEMM_ERR_TOO_LARGE = -9
ARRAY_FLOATS = 1 << 24          # the fixed array: 16,777,216 floats


@pytest.fixture(scope="module")
def noalloc():
    sg.build()
    sg.force_kernel(sg.KERNEL_AUTO)
    fn = sg.lib().sgemm_noalloc
    fn.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]
    fn.restype = ctypes.c_int
    return fn


def _operands(M, N, K, seed):
    A = synth.matrix(M, K, seed=seed, stream=0, dist="normal")
    B = synth.matrix(K, N, seed=seed, stream=1, dist="normal")
    C0 = synth.matrix(M, N, seed=seed, stream=2, dist="normal")
    return A, B, C0


def _call(noalloc, dA, dB, dC, alpha, beta, stream=None):
    M, K = dA.shape
    N = dB.shape[1]
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, dC.data_ptr(), N, s)


def _compare_one(noalloc, M, N, K, alpha, beta, seed):
    """One sgemm_noalloc call against the oracle and against sgemm()."""
    A, B, C0 = _operands(M, N, K, seed)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    want = torch.from_numpy(C0).cuda()
    got = want.clone()
    kid = sg.select_kernel(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                           got.data_ptr(), N)
    assert kid == sg.KERNEL_FFMA_TMA, "these shapes must take the scratch-using kernel"
    rc = _call(noalloc, dA, dB, got, alpha, beta)
    assert rc == sg.OK, sg.status_string(rc)
    assert sg.status() == sg.OK
    sg.sgemm(dA, dB, want, alpha, beta)
    assert sg.status() == sg.OK
    got_h, want_h = got.cpu().numpy(), want.cpu().numpy()
    ref = oracle.sgemm(A, B, C0, alpha=alpha, beta=beta)
    err = normwise_err(got_h, ref, A, B, K, alpha, beta, C0)
    assert err <= GATE, f"sgemm_noalloc against the oracle: {err:.3e}"
    err = normwise_err(got_h, want_h, A, B, K, alpha, beta, C0)
    assert err <= GATE, f"sgemm_noalloc differs from sgemm: {err:.3e}"
    return got_h, want_h


def test_matches_oracle_and_sgemm_on_two_calls_in_a_row(noalloc):
    # The first call fills more of the array than the second reads.
    _compare_one(noalloc, 1000, 700, 1500, 1.0, 0.5, seed=41)
    _compare_one(noalloc, 300, 516, 260, -0.75, 0.0, seed=42)


def test_full_array_runs_the_tail_as_whole_tiles(noalloc):
    # M = K = 4096: A^T fills the array, so the partial tiles of a divided
    # tail have no room.  At N = 512 the 4096 x 512 output is a few hundred
    # tiles, less than one wave of resident CTAs, which sgemm() (whose
    # workspace grows) divides by work along K; sgemm_noalloc must run the
    # tiles whole.
    M = K = 4096
    assert K * M == ARRAY_FLOATS
    got, want = _compare_one(noalloc, M, 512, K, 1.0, 0.25, seed=43)
    # the two entry points summed the k-steps in different orders
    assert not np.array_equal(got, want)


def test_allocates_nothing(noalloc):
    M, N, K = 1000, 700, 1500
    A, B, C0 = _operands(M, N, K, seed=44)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    # set-up call (module load, array address)
    assert _call(noalloc, dA, dB, dC, 1.0, 0.0) == sg.OK
    stream = torch.cuda.Stream()
    # no workspace anywhere: an sgemm()-style call would have to allocate one
    assert sg.release_workspaces() == sg.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _call(noalloc, dA, dB, dC, 1.0, 0.0, stream=stream) == sg.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0, f"sgemm_noalloc took {free0 - free1} bytes of device memory"
    got = dC.cpu().numpy()
    # the same measurement sees sgemm()'s workspace (4 * K * M bytes of A^T)
    rc = sg.lib().sgemm(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, dC.data_ptr(), N,
                        stream.cuda_stream)
    assert rc == sg.OK
    torch.cuda.synchronize()
    free2, _ = torch.cuda.mem_get_info()
    assert free1 - free2 >= 4 * K * M, "the free-memory measurement did not see sgemm()'s workspace"
    assert sg.status() == sg.OK
    ref = oracle.sgemm(A, B, alpha=1.0, beta=0.0)
    assert normwise_err(got, ref, A, B, K) <= GATE


@pytest.mark.parametrize("forced", [sg.KERNEL_TF32X3, sg.KERNEL_TF32, sg.KERNEL_BF16])
def test_forced_tensor_core_kernel_is_refused(noalloc, forced):
    M, N, K = 300, 256, 260
    A, B, C0 = _operands(M, N, K, seed=45)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    prev = sg.force_kernel(forced)
    try:
        rc = _call(noalloc, dA, dB, dC, 1.0, 0.5)
    finally:
        sg.force_kernel(prev)
    assert rc == sg.ERR_BAD_ARG
    torch.cuda.synchronize()
    assert np.array_equal(dC.cpu().numpy(), C0), "a refused call changed C"


def test_refuses_problems_beyond_the_array(noalloc):
    # K * round_up(M, 4) = 4100 * 4100 > 16,777,216: refused before any
    # launch.  Real device buffers, so a regression gives a wrong result
    # rather than a bad address.
    M = N = K = 4100
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    dC = torch.full((M, N), 3.0, device="cuda")
    assert _call(noalloc, dA, dB, dC, 1.0, 0.0) == SGEMM_ERR_TOO_LARGE
    assert "fixed scratch" in sg.status_string(SGEMM_ERR_TOO_LARGE)
    torch.cuda.synchronize()
    assert bool((dC == 3.0).all()), "a refused call changed C"
    assert sg.status() == sg.OK
