"""sgemm calls captured in a CUDA graph and replayed.

A decode step is typically launched from a CUDA graph, so the library's calls
must capture: after one eager call of the same shape on the stream (device
set-up, workspace sized), a captured call enqueues its kernels and nothing
else, and a replay recomputes C from the operands' current contents.  A
captured call that would have to grow the stream's workspace is refused with
SGEMM_ERR_CAPTURE instead of allocating inside the graph.
"""

import numpy as np
import pytest

from gpu_util import GATE, make_inputs, normwise_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402
import oracle  # noqa: E402


@pytest.mark.parametrize("M,N,K,tc", [(16, 14336, 4096, False), (4, 1000, 700, False),
                                      (1000, 1000, 1000, False), (300, 516, 260, False),
                                      (256, 512, 384, True), (256, 512, 384, sg.MODE_TF32),
                                      (256, 512, 384, sg.MODE_BF16)])
def test_capture_and_replay(M, N, K, tc):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + N + K, beta=0.5)
    s = torch.cuda.Stream()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    eager = dC.clone()
    with torch.cuda.stream(s):
        sg.sgemm(dA, dB, eager, 1.25, 0.5, stream=s, tensor_cores=tc)
    s.synchronize()
    assert sg.status(s) == sg.OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sg.sgemm(dA, dB, dC, 1.25, 0.5, stream=s, tensor_cores=tc)
    # capture enqueued nothing: C still holds C0
    assert np.array_equal(dC.cpu().numpy(), C0)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert sg.status(s) == sg.OK
    got = dC.cpu().numpy()
    assert np.array_equal(got, eager.cpu().numpy()), "replay differs from the eager call"
    inputs = {sg.MODE_TF32: "tf32", sg.MODE_BF16: "bf16"}.get(sg._mode(tc), "fp32")
    ref = oracle.sgemm(A, B, C0, alpha=1.25, beta=0.5, inputs=inputs)
    assert normwise_err(got, ref, A, B, K, 1.25, 0.5, C0) <= GATE
    # a second replay reads the operands' new contents
    A2 = np.ascontiguousarray(A[::-1])
    dA.copy_(torch.from_numpy(A2))
    dC.copy_(torch.from_numpy(C0))
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    ref2 = oracle.sgemm(A2, B, C0, alpha=1.25, beta=0.5, inputs=inputs)
    assert normwise_err(dC.cpu().numpy(), ref2, A2, B, K, 1.25, 0.5, C0) <= GATE


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_capture_refuses_to_grow_the_workspace():
    torch.cuda.synchronize()
    sg.release_workspaces()        # streams come from a pool: start from no workspace
    s = torch.cuda.Stream()
    dA = torch.randn(300, 260, device="cuda")
    dB = torch.randn(260, 516, device="cuda")
    dC = torch.empty(300, 516, device="cuda")
    with torch.cuda.stream(s):
        sg.sgemm(dA, dB, dC, 1.0, 0.0, stream=s)          # sizes the workspace for this shape
    s.synchronize()
    big_A = torch.randn(2000, 3000, device="cuda")
    big_B = torch.randn(3000, 516, device="cuda")
    big_C = torch.empty(2000, 516, device="cuda")
    g = torch.cuda.CUDAGraph()
    with pytest.raises(sg.SgemmError) as ei:
        with torch.cuda.graph(g, stream=s):
            sg.sgemm(big_A, big_B, big_C, 1.0, 0.0, stream=s)
    assert ei.value.code == sg.ERR_CAPTURE


@pytest.mark.parametrize("captured", [False, True])
def test_chained_decode_products_see_each_others_results(captured):
    # Each decode kernel may become resident while the kernel before it on
    # the stream is still running and waits for it before its first copy.
    # Chains C1 = A0 B1, C2 = C1 B2 (the second product reads the first one's
    # output as A), repeated back to back with C1 and C2 reset to NaN before
    # each chain: a product that read its A too early would see NaN.  Small
    # integers keep every sum exact, so each link must match the oracle's
    # chain bit for bit.
    M, K0, K1, N = 16, 4096, 512, 4096
    rng = np.random.default_rng(61)
    A0 = rng.integers(-1, 2, (M, K0)).astype(np.float32)
    B1 = rng.integers(-1, 2, (K0, K1)).astype(np.float32)
    B2 = rng.integers(-1, 2, (K1, N)).astype(np.float32)
    C1_ref = oracle.sgemm(A0, B1, alpha=1.0, beta=0.0)
    C2_ref = oracle.sgemm(C1_ref.astype(np.float32), B2, alpha=1.0, beta=0.0)
    assert np.abs(C2_ref).max() < 2 ** 24
    s = torch.cuda.Stream()
    dA0, dB1, dB2 = (torch.from_numpy(x).cuda() for x in (A0, B1, B2))
    chains = 6
    C1 = [torch.empty((M, K1), device="cuda") for _ in range(chains)]
    C2 = [torch.empty((M, N), device="cuda") for _ in range(chains)]
    assert sg.select_kernel(M, K1, K0, 1.0, dA0.data_ptr(), K0, dB1.data_ptr(), K1, 0.0,
                            C1[0].data_ptr(), K1) == sg.KERNEL_DECODE
    assert sg.select_kernel(M, N, K1, 1.0, C1[0].data_ptr(), K1, dB2.data_ptr(), N, 0.0,
                            C2[0].data_ptr(), N) == sg.KERNEL_DECODE

    def run():
        for i in range(chains):
            sg.sgemm(dA0, dB1, C1[i], 1.0, 0.0, stream=s)
            sg.sgemm(C1[i], dB2, C2[i], 1.0, 0.0, stream=s)

    with torch.cuda.stream(s):
        run()                                  # set-up calls
    s.synchronize()
    for t in C1 + C2:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    if captured:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run()
        with torch.cuda.stream(s):
            g.replay()
    else:
        with torch.cuda.stream(s):
            run()
    s.synchronize()
    assert sg.status(s) == sg.OK
    for i in range(chains):
        assert np.array_equal(C1[i].cpu().numpy(), C1_ref.astype(np.float32)), f"chain {i}: C1"
        assert np.array_equal(C2[i].cpu().numpy(), C2_ref.astype(np.float32)), f"chain {i}: C2"
