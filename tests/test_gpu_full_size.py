"""Whole-matrix parity at the full benchmark sizes, through the C ABI.

Every element of C is compared with the fp64 oracle, which is the GEMM
definition of "GPU GEMM 优化完全拆解（一）", section "什么是 GEMM":

  - 4092^3 on small integers in [-4, 4] (alpha = 1, beta = 0.5): bit-exact,
    because every partial sum is an integer below 2^24;
  - 8192^3, normal(0, 1) from seed 2, on all four arithmetics: sgemm (FFMA)
    and sgemm_3xtf32 against the oracle on the operands themselves,
    sgemm_tf32 / sgemm_bf16 against the oracle on the rounded operands;
  - the prefill GEMMs QKV 8192x12288x4096, FFN-up 8192x14336x4096 and
    FFN-down 8192x4096x14336 (activations normal(0, 1), weights
    normal(0, 0.02), seed 4) on sgemm.

Each launch is the one bench.py times for that shape (the library's own
choice of kernel and tile configuration).  The 8192^3 oracle result is
computed once and shared by the FFMA, 3xTF32 and accuracy-ratio tests.

The accuracy-ratio test is the discrimination check for the 3xTF32 path:
over the whole 8192^3 matrix its error must stay within 4x the FFMA path's
error on the same operands, i.e. the tensor-core variant keeps FP32
accuracy (one TF32 term would be two orders of magnitude worse).
"""

import numpy as np
import pytest

import oracle
import synth
from gpu_util import GATE, product_err, run_checked

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    sg.build()
    sg.force_kernel(sg.KERNEL_AUTO)
    yield


@pytest.fixture(scope="module")
def w8192():
    """Operands of the 8192^3 workload and the oracle's full result (once)."""
    A, B, _, w = synth.workload_inputs("sgemm_8192")
    ref = oracle.sgemm(A, B, None, alpha=w["alpha"], beta=w["beta"])
    yield A, B, w, ref


def _nan_c(w):
    # beta = 0: C must not be read, so it starts as NaN
    return np.full((w["M"], w["N"]), np.nan, np.float32)


def test_workload_4092_int_exact_all_rows():
    A = synth.matrix(4092, 4092, seed=1, stream=0, dist="int")
    B = synth.matrix(4092, 4092, seed=1, stream=1, dist="int")
    C0 = synth.matrix(4092, 4092, seed=1, stream=2, dist="int")
    _, chosen = run_checked(sg, A, B, C0, 1.0, 0.5, exact=True)
    assert chosen == sg.KERNEL_FFMA_TMA


@pytest.mark.parametrize("mode", [sg.MODE_FP32, sg.MODE_3XTF32])
def test_workload_8192_full(w8192, mode):
    A, B, w, ref = w8192
    _, chosen = run_checked(sg, A, B, _nan_c(w), w["alpha"], w["beta"], tensor_cores=mode,
                            ref=ref)
    assert chosen == {sg.MODE_FP32: sg.KERNEL_FFMA_TMA, sg.MODE_3XTF32: sg.KERNEL_TF32X3}[mode]


@pytest.mark.parametrize("mode,inputs,kernel", [(sg.MODE_TF32, "tf32", sg.KERNEL_TF32),
                                                (sg.MODE_BF16, "bf16", sg.KERNEL_BF16)])
def test_workload_8192_reduced_precision_full(w8192, mode, inputs, kernel):
    A, B, w, _ = w8192
    ref = oracle.sgemm(A, B, None, alpha=w["alpha"], beta=w["beta"], inputs=inputs)
    _, chosen = run_checked(sg, A, B, _nan_c(w), w["alpha"], w["beta"], tensor_cores=mode,
                            ref=ref)
    assert chosen == kernel


def test_workload_8192_3xtf32_error_within_4x_ffma(w8192):
    A, B, w, ref = w8192
    K = w["K"]
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    errs = {}
    for mode in (sg.MODE_FP32, sg.MODE_3XTF32):
        dC = torch.empty((w["M"], w["N"]), device="cuda")
        sg.sgemm(dA, dB, dC, w["alpha"], w["beta"], tensor_cores=mode)
        assert sg.status() == sg.OK
        errs[mode] = product_err(dC.cpu().numpy(), ref, A, B, K)
        del dC
    assert errs[sg.MODE_FP32] <= GATE and errs[sg.MODE_3XTF32] <= GATE, errs
    assert errs[sg.MODE_3XTF32] <= 4 * errs[sg.MODE_FP32], \
        f"3xTF32 error {errs[sg.MODE_3XTF32]:.3e} > 4 x FFMA error {errs[sg.MODE_FP32]:.3e}"


@pytest.mark.parametrize("name", ["prefill_qkv", "prefill_up", "prefill_down"])
def test_workload_prefill_full(name):
    A, B, C0, w = synth.workload_inputs(name)
    C0 = _nan_c(w) if C0 is None else C0
    _, chosen = run_checked(sg, A, B, C0, w["alpha"], w["beta"])
    assert chosen == sg.KERNEL_FFMA_TMA
