"""sgemm_host: the product for operands in host memory, through the C ABI.

The library copies B and row panels of A and C to the device, multiplies each
panel as it arrives and copies its rows of C back, overlapping the three.
These tests check the result against the fp64 oracle (the normwise gate, or
bit-exact where the arithmetic is exact) on single- and multi-panel shapes
with a ragged last panel, row-strided host buffers whose gap columns hold
canaries, pinned and pageable memory, every arithmetic mode, the quick paths
and back-to-back calls that grow the library's device buffer.
"""

import numpy as np
import pytest

import oracle
from gpu_util import CANARY_BITS, GATE, make_inputs, normwise_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    sg.build()
    prev = sg.host_set_panels(0)
    yield
    sg.host_set_panels(prev)


class HostMatrix:
    """A rows x cols matrix in host memory with row stride ld >= cols; the gap
    columns hold canaries."""

    def __init__(self, X, ld=None, pinned=True):
        rows, cols = X.shape
        self.ld = cols if ld is None else ld
        buf = np.full((rows, max(self.ld, 1)), CANARY_BITS, dtype=np.uint32).view(np.float32)
        buf[:, :cols] = X
        t = torch.from_numpy(buf)
        self.buf = t.pin_memory() if pinned else t
        self.view = self.buf[:, :cols]
        self.cols = cols

    def matrix(self):
        return self.buf.numpy()[:, :self.cols].copy()

    def gaps_intact(self):
        g = self.buf.numpy()[:, self.cols:].view(np.uint32)
        return bool((g == CANARY_BITS).all())


def run_host(A, B, C0, alpha, beta, *, lds=(None, None, None), pinned=True, mode=False,
             panels=0, exact=False):
    M, K = A.shape
    N = B.shape[1]
    ha, hb = HostMatrix(A, lds[0], pinned), HostMatrix(B, lds[1], pinned)
    hc = HostMatrix(C0, lds[2], pinned)
    prev = sg.host_set_panels(panels)
    try:
        stream = torch.cuda.current_stream()
        sg.sgemm_host(ha.view, hb.view, hc.view, alpha, beta, stream=stream, tensor_cores=mode)
        st = sg.status(stream)
    finally:
        sg.host_set_panels(prev)
    assert st == sg.OK, sg.status_string(st)
    C = hc.matrix()
    assert hc.gaps_intact(), "a write landed in C's gap columns"
    assert np.array_equal(ha.matrix(), A) and np.array_equal(hb.matrix(), B)
    inputs = {sg.MODE_TF32: "tf32", sg.MODE_BF16: "bf16"}.get(sg._mode(mode), "fp32")
    ref = oracle.sgemm(A, B, C0 if beta != 0.0 else None, alpha=alpha, beta=beta, inputs=inputs)
    if exact:
        assert np.array_equal(C, ref), f"not bit-exact: max |diff| {np.abs(C - ref).max()}"
        return 0.0
    err = normwise_err(C, ref, A, B, K, alpha, beta, C0)
    assert err <= GATE, f"normwise error {err:.3e} above {GATE}"
    return err


@pytest.mark.parametrize("panels", [0, 1, 2, 3, 5])
def test_panels_ragged_and_strided(panels):
    M, N, K = 1000, 700, 300
    A, B, C0 = make_inputs(M, N, K, "normal", seed=71, beta=0.5)
    run_host(A, B, C0, 1.5, 0.5, lds=(K + 3, N + 5, N + 2), panels=panels)


@pytest.mark.parametrize("lds", [(None, None, None), (364, 704, 700), (400, 800, 702)])
def test_linear_and_pitched_copies(lds):
    # equal host and device strides move each operand with one linear copy
    # (gaps included on the way up, never on the way back); wide gaps and
    # strides the kernels cannot take go through pitched copies
    M, N, K = 700, 700, 300
    A, B, C0 = make_inputs(M, N, K, "normal", seed=90, beta=0.5)
    run_host(A, B, C0, 1.0, 0.5, lds=lds, panels=3)


@pytest.mark.parametrize("M,N,K,panels", [(700, 300, 1500, 2), (900, 260, 2500, 3),
                                           (600, 200, 4100, 4)])
def test_first_panel_in_k_ranges(M, N, K, panels):
    # with several panels and K >= 1024 the first panel is multiplied in 2 or 4
    # K-ranges while B is still arriving; beta != 0 and beta == 0 both
    for beta, seed in ((0.5, 91), (0.0, 92)):
        A, B, C0 = make_inputs(M, N, K, "normal", seed=seed + K, beta=beta)
        run_host(A, B, C0, 0.75, beta, panels=panels, lds=(K + 4, N, N))


@pytest.mark.parametrize("mode", [sg.MODE_3XTF32, sg.MODE_BF16])
def test_first_panel_in_k_ranges_tensor_cores(mode):
    # the K-ranged first panel with the tensor-core arithmetics (each range is
    # one call of that entry point, so the rounded-operand contracts hold)
    M, N, K = 640, 384, 2048
    A, B, C0 = make_inputs(M, N, K, "normal", seed=94 + mode, beta=0.5)
    run_host(A, B, C0, 1.0, 0.5, mode=mode, panels=2)


def test_first_panel_in_k_ranges_small_integers_exact():
    # partial sums of small integers are exact, so splitting K changes nothing
    M, N, K = 800, 300, 2100
    A, B, C0 = make_inputs(M, N, K, "int", seed=93, beta=1.0)
    run_host(A, B, C0, 1.0, 1.0, panels=3, exact=True)


def test_default_panel_count_on_a_large_square():
    # the 4092^3 benchmark shape splits into several panels by default; every
    # row is checked against the oracle
    M = N = K = 4092
    assert sg.host_panel_rows(M, N, K) < M
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=72, beta=0.5)
    run_host(A, B, C0, 1.0, 0.5)


def test_small_integers_exact_across_panels():
    M, N, K = 777, 515, 260
    A, B, C0 = make_inputs(M, N, K, "int", seed=73, beta=1.0)
    run_host(A, B, C0, 1.0, 1.0, panels=4, exact=True)


def test_beta_zero_does_not_read_host_c():
    M, N, K = 600, 400, 200
    A, B, _ = make_inputs(M, N, K, "uniform", seed=74)
    C0 = np.full((M, N), np.nan, dtype=np.float32)
    run_host(A, B, C0, 1.0, 0.0, panels=3)


def test_pageable_memory():
    M, N, K = 513, 300, 257
    A, B, C0 = make_inputs(M, N, K, "normal", seed=75, beta=-1.0)
    run_host(A, B, C0, 0.75, -1.0, pinned=False, panels=2, lds=(K, N + 1, N))


@pytest.mark.parametrize("M", [1, 5, 16])
def test_decode_shapes(M):
    N, K = 3000, 700
    A, B, C0 = make_inputs(M, N, K, "normal", seed=76 + M, beta=0.25)
    run_host(A, B, C0, 1.0, 0.25)


@pytest.mark.parametrize("mode", [sg.MODE_3XTF32, sg.MODE_TF32, sg.MODE_BF16])
def test_tensor_core_modes(mode):
    M, N, K = 640, 384, 512
    A, B, C0 = make_inputs(M, N, K, "normal", seed=80 + mode, beta=0.5)
    # TF32 / BF16: the reduced-precision contracts (the oracle on rounded operands)
    run_host(A, B, C0, 1.0, 0.5, mode=mode, panels=2)


def test_quick_paths_are_exact():
    M, N, K = 300, 200, 100
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=84, beta=0.5)
    run_host(A, B, C0, 0.0, 0.5, exact=True)                   # alpha = 0: C = beta*C
    run_host(A[:, :0], B[:0, :], C0, 2.0, 0.5, exact=True)     # K = 0


def test_back_to_back_calls_grow_the_buffer():
    # small then large then small on one stream: the device buffer grows in
    # stream order and the later calls see their own operands
    for (M, N, K), seed in (((200, 150, 90), 85), ((1500, 1100, 700), 86), ((260, 140, 60), 87)):
        A, B, C0 = make_inputs(M, N, K, "uniform", seed=seed, beta=0.5)
        run_host(A, B, C0, 1.0, 0.5, panels=0 if M < 1000 else 3)


def test_ordered_with_other_work_on_the_stream():
    # work enqueued on the stream after the call (a copy of host C to the
    # device and back) sees the finished result without any host wait between
    M, N, K = 900, 500, 400
    A, B, C0 = make_inputs(M, N, K, "normal", seed=88, beta=0.0)
    ha, hb, hc = (HostMatrix(X) for X in (A, B, np.zeros((M, N), np.float32)))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        prev = sg.host_set_panels(3)
        try:
            sg.sgemm_host(ha.view, hb.view, hc.view, 1.0, 0.0, stream=stream)
        finally:
            sg.host_set_panels(prev)
        d = hc.view.to("cuda", non_blocking=True)   # ordered after the call on `stream`
        back = d.cpu()
    assert sg.status(stream) == sg.OK
    ref = oracle.sgemm(A, B, None, alpha=1.0, beta=0.0)
    assert normwise_err(back.numpy(), ref, A, B, K) <= GATE
    assert normwise_err(hc.matrix(), ref, A, B, K) <= GATE


def test_capture_is_refused():
    M, N, K = 64, 64, 64
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=89)
    ha, hb, hc = (HostMatrix(X) for X in (A, B, np.zeros((M, N), np.float32)))
    s = torch.cuda.Stream()
    x = torch.zeros(4, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    rc = None
    with torch.cuda.graph(g, stream=s):
        x.add_(1.0)
        rc = sg.lib().sgemm_host(M, N, K, 1.0, ha.view.data_ptr(), K, hb.view.data_ptr(), N, 0.0,
                                 hc.view.data_ptr(), N, 0, s.cuda_stream)
    assert rc == sg.ERR_CAPTURE
