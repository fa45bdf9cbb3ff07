"""Parity of the CUDA library with the fp64 oracle, through the C ABI.

Every case runs on padded device buffers with NaN canaries in the gaps and
guards (see gpu_util.Padded) and checks: the kernel the library chose, the
status word, that nothing outside C's elements changed, and the oracle gate
max|C - C_ref| / (K * max|A| * max|B|) <= 1e-6, or bit-exact equality on
small-integer inputs and on the closed forms.
"""

import itertools

import numpy as np
import pytest

import synth
from gpu_util import GATE, make_inputs, run_checked

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import dense_fp32_matrix_row_gb300 as sg  # noqa: E402

TMA, GEN, DEC = sg.KERNEL_FFMA_TMA, sg.KERNEL_FFMA_GENERIC, sg.KERNEL_DECODE


@pytest.fixture(scope="module", autouse=True)
def built():
    sg.build()
    sg.force_kernel(sg.KERNEL_AUTO)
    yield


def kernels_for(M):
    return [TMA, GEN] + ([DEC] if M <= 16 else [])


# ---------------------------------------------------------------- brute force grid
GRID = [1, 5, 16, 17, 33, 128, 129]


@pytest.mark.parametrize("M,N,K", list(itertools.product(GRID, GRID, GRID)))
def test_grid_all_kernels(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M * 1000 + N * 10 + K, beta=0.75)
    for k in kernels_for(M):
        _, chosen = run_checked(sg, A, B, C0, 1.25, 0.75, kernel=k)
        assert chosen == k


@pytest.mark.parametrize("M,N,K", [(300, 260, 100), (129, 385, 77), (257, 129, 1000),
                                   (511, 513, 31), (640, 384, 4097), (1, 2000, 3000)])
def test_multi_tile_ragged(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + N + K, beta=-0.5)
    for k in kernels_for(M):
        _, chosen = run_checked(sg, A, B, C0, 0.5, -0.5, kernel=k)
        assert chosen == k


DEC_M = [1, 2, 3, 4, 5, 8, 9, 12, 16]
DEC_N = [1, 3, 129, 1000]
DEC_K = [1, 65, 700, 1028, 4097]


@pytest.mark.parametrize("M,N,K", list(itertools.product(DEC_M, DEC_N, DEC_K)))
def test_decode_shapes(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=7 * M + N + K, beta=1.0, sigma_b=0.02)
    _, chosen = run_checked(sg, A, B, C0, 1.0, 1.0)
    assert chosen == DEC


# The outer-product tile with M = 9..16 rows and long K: clusters of up to
# 16 blocks (non-portable sizes), ragged last K slices, integer data so that
# any misplaced or dropped k-step shows exactly.
@pytest.mark.parametrize("M,K", [(9, 436), (16, 3364), (12, 6720), (16, 6724), (13, 8192)])
def test_decode_slice_limits(M, K):
    N = 300
    A, B, C0 = make_inputs(M, N, K, "int", seed=M + K, beta=-2.0)
    _, chosen = run_checked(sg, A, B, C0, 3.0, -2.0, exact=True)
    assert chosen == DEC


# ---------------------------------------------------------------- exactness
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (4, 14336, 4096), (300, 200, 1000),
                                   (16, 129, 5000)])
def test_small_integers_exact(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "int", seed=3, beta=-2.0)
    for k in kernels_for(M):
        run_checked(sg, A, B, C0, 3.0, -2.0, kernel=k, exact=True)


@pytest.mark.parametrize("k", [TMA, GEN, DEC])
def test_identity_and_permutation_exact(k):
    n = 16 if k == DEC else 200
    B = synth.matrix(n, 150, seed=5, stream=1, dist="normal")
    eye = np.eye(n, dtype=np.float32)
    nan = np.full((n, 150), np.nan, dtype=np.float32)
    run_checked(sg, eye, B, nan, 1.0, 0.0, kernel=k, exact=True)
    p = np.random.default_rng(5).permutation(n)
    P = np.zeros((n, n), dtype=np.float32)
    P[np.arange(n), p] = 1.0
    run_checked(sg, P, B, nan, 1.0, 0.0, kernel=k, exact=True)


@pytest.mark.parametrize("k", [TMA, GEN, DEC])
def test_rank1_exact(k):
    M, N, K = (9 if k == DEC else 130), 70, 999
    u = (np.arange(M) % 5 - 2).astype(np.float32)
    v = (np.arange(N) % 7 - 3).astype(np.float32)
    A = np.repeat(u[:, None], K, axis=1).astype(np.float32)
    B = np.repeat(v[None, :], K, axis=0).astype(np.float32)
    run_checked(sg, A, B, np.full((M, N), np.nan, np.float32), 1.0, 0.0, kernel=k, exact=True)


# ---------------------------------------------------------------- alpha / beta
@pytest.mark.parametrize("k", [TMA, GEN, DEC])
def test_alpha_beta_semantics(k):
    M = 12 if k == DEC else 70
    N, K = 45, 33
    A, B, C0 = make_inputs(M, N, K, "int", seed=11, beta=1.0)
    for alpha, beta in [(1.0, 0.0), (1.0, 1.0), (1.0, 0.5), (-1.0, 2.0), (0.0, 3.0), (0.0, 0.0),
                        (2.0, -1.0)]:
        c = C0 if beta != 0.0 else np.full((M, N), np.nan, np.float32)
        run_checked(sg, A, B, c, alpha, beta, kernel=k, exact=True)


def test_k_zero_and_empty():
    for (M, N) in [(5, 7), (300, 3)]:
        A = np.zeros((M, 0), np.float32)
        B = np.zeros((0, N), np.float32)
        C0 = synth.matrix(M, N, seed=1, stream=2)
        _, chosen = run_checked(sg, A, B, C0, 1.0, 0.25)
        assert chosen == sg.KERNEL_SCALE_C
        _, chosen = run_checked(sg, A, B, np.full((M, N), np.nan, np.float32), 1.0, 0.0)
        assert chosen == sg.KERNEL_SCALE_C
    for (M, N, K) in [(0, 5, 5), (5, 0, 5), (0, 0, 0)]:
        A, B, C0 = make_inputs(M, N, K, beta=1.0)
        _, chosen = run_checked(sg, A, B, C0, 1.0, 1.0)
        assert chosen == sg.KERNEL_NONE


def test_nan_in_inputs_propagates():
    M, N, K = 64, 64, 64
    A, B, _ = make_inputs(M, N, K, "uniform", seed=2)
    A[3, 5] = np.nan
    for k in (TMA, GEN):
        from gpu_util import Padded
        pa, pb = Padded(A), Padded(B)
        pc = Padded(np.zeros((M, N), np.float32))
        sg.force_kernel(k)
        try:
            sg.sgemm(pa.view, pb.view, pc.view, 1.0, 0.0)
            assert sg.status() == sg.OK
        finally:
            sg.force_kernel(sg.KERNEL_AUTO)
        C = pc.matrix()
        assert np.isnan(C[3]).all() and np.isfinite(np.delete(C, 3, axis=0)).all()


# ---------------------------------------------------------------- layouts
@pytest.mark.parametrize("lds,offsets,expect", [
    ((170, 53, 61), (0, 0, 0), GEN),       # ld % 4 != 0 everywhere
    ((168, 52, 61), (0, 0, 0), TMA),       # A, B TMA-able, C scalar epilogue
    ((168, 52, 56), (0, 0, 1), TMA),       # C misaligned by one float
    ((168, 52, 56), (1, 0, 0), TMA),       # A misaligned: read through its transposed copy
    ((170, 52, 56), (0, 0, 0), TMA),       # lda % 4 != 0: likewise
    ((168, 52, 56), (0, 2, 0), GEN),       # B misaligned
    ((168, 53, 56), (0, 0, 0), GEN),       # ldb % 4 != 0
    ((164, 48, 48), (0, 0, 0), TMA),       # dense
])
def test_leading_dims_and_alignment(lds, offsets, expect):
    # more than 2^21 multiply-adds, so the choice is not the tiny-product one
    M, N, K = 300, 48, 164
    A, B, C0 = make_inputs(M, N, K, "normal", seed=13, beta=0.5)
    _, chosen = run_checked(sg, A, B, C0, 1.0, 0.5, lds=lds, offsets=offsets)
    assert chosen == expect


def test_decode_layouts():
    M, N, K = 7, 300, 500
    A, B, C0 = make_inputs(M, N, K, "normal", seed=17, beta=0.5)
    for lds, offsets in [((503, 301, 300), (0, 0, 0)), ((500, 304, 300), (1, 1, 1)),
                         ((512, 304, 301), (0, 0, 3))]:
        _, chosen = run_checked(sg, A, B, C0, 1.0, 0.5, lds=lds, offsets=offsets)
        assert chosen == DEC


def test_tall_and_wide_extremes():
    for (M, N, K) in [(70000, 4, 8), (4, 70000, 8), (17, 5, 70000)]:
        A, B, C0 = make_inputs(M, N, K, "uniform", seed=19, beta=0.0)
        run_checked(sg, A, B, C0, 1.0, 0.0)


# ---------------------------------------------------------------- behaviour
def test_deterministic_and_streams():
    M, N, K = 513, 257, 1031
    A, B, _ = make_inputs(M, N, K, "normal", seed=23)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    s = torch.cuda.Stream()
    outs = []
    for M_ in (M, 9):
        for _ in range(2):
            C = torch.empty((M_, N), device="cuda")
            with torch.cuda.stream(s):
                sg.sgemm(dA[:M_], dB, C, 1.0, 0.0, stream=s)
            assert sg.status(s) == sg.OK
            outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[2], outs[3])


def test_workspace_release_and_regrow():
    A, B, C0 = make_inputs(300, 200, 260, "int", seed=31, beta=1.0)
    run_checked(sg, A, B, C0, 1.0, 1.0, exact=True)
    assert sg.release_workspaces() == sg.OK
    A, B, C0 = make_inputs(700, 90, 1100, "int", seed=32, beta=0.0)
    run_checked(sg, A, B, C0, 1.0, 0.0, exact=True)   # grows a fresh workspace


def test_rejected_arguments_raise():
    A = torch.zeros((4, 4), device="cuda")
    with pytest.raises(ValueError):
        sg.sgemm(A, torch.zeros((5, 4), device="cuda"), torch.zeros((4, 4), device="cuda"))
    with pytest.raises(sg.SgemmError) as e:
        sg.sgemm(A, A, A)              # C aliases A
    assert e.value.code == sg.ERR_ALIAS
    with pytest.raises(TypeError):
        sg.sgemm(A.double(), A, torch.zeros((4, 4), device="cuda"))


def test_bounded_wait_times_out_and_context_survives():
    assert sg.status() == sg.OK
    assert sg.selftest_wait(2_000_000) == sg.OK       # 2 ms on a barrier nothing completes
    assert sg.status() == sg.ERR_TIMEOUT
    assert sg.status() == sg.OK                       # cleared
    A, B, C0 = make_inputs(130, 70, 90, "int", seed=29, beta=1.0)
    run_checked(sg, A, B, C0, 1.0, 1.0, exact=True)   # the context still works


# ---------------------------------------------------------------- full-size workloads
# (the 4092^3 integer case, 8192^3 and the prefill GEMMs: test_gpu_full_size.py)
@pytest.mark.parametrize("name", ["sgemm_128", "sgemm_128_int", "decode_m1", "decode_m4",
                                  "decode_m16"])
def test_workload_full(name):
    A, B, C0, w = synth.workload_inputs(name)
    if C0 is None:
        C0 = np.full((w["M"], w["N"]), np.nan, np.float32)
    run_checked(sg, A, B, C0, w["alpha"], w["beta"], exact=name.endswith("_int"))


def test_workload_4092_full():
    """4092^3, alpha=1, beta=0.5: every output against the oracle."""
    A, B, C0, w = synth.workload_inputs("sgemm_4092")
    err, chosen = run_checked(sg, A, B, C0, w["alpha"], w["beta"])
    assert chosen == TMA and err <= GATE


# ---------------------------------------------------------------- 3xTF32 tensor-core path
TF = sg.KERNEL_TF32X3


@pytest.mark.parametrize("M,N,K", [(17, 5, 3), (128, 256, 16), (129, 257, 33), (300, 260, 100),
                                   (255, 513, 1000), (1000, 300, 4097), (17, 1, 1)])
def test_tf32x3_shapes(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M * 7 + N + K, beta=0.5)
    _, chosen = run_checked(sg, A, B, C0, 1.25, 0.5, tensor_cores=True)
    assert chosen == TF


def test_tf32x3_small_integers_exact():
    # integers in [-4, 4] are exact TF32 numbers (lo = 0) and every partial sum
    # stays below 2^24, so the tensor-core result is exact
    A, B, C0 = make_inputs(300, 200, 1000, "int", seed=5, beta=-2.0)
    run_checked(sg, A, B, C0, 3.0, -2.0, tensor_cores=True, exact=True)


def test_tf32x3_alpha_beta_and_layouts():
    M, N, K = 70, 45, 33
    A, B, C0 = make_inputs(M, N, K, "int", seed=12, beta=1.0)
    for alpha, beta in [(1.0, 0.0), (1.0, 1.0), (-1.0, 0.5), (0.0, 3.0), (2.0, -1.0)]:
        c = C0 if beta != 0.0 else np.full((M, N), np.nan, np.float32)
        run_checked(sg, A, B, c, alpha, beta, tensor_cores=True, exact=True)
    for lds, offsets in [((37, 47, 46), (1, 3, 1)), ((40, 48, 48), (0, 0, 0))]:
        run_checked(sg, A, B, C0, 1.0, 1.0, lds=lds, offsets=offsets, tensor_cores=True,
                    exact=True)


def test_tf32x3_is_three_term():
    """Inputs with 24 significant bits: one TF32 product keeps 11, so a 1xTF32
    result misses the 1e-6 gate here by an order of magnitude; the 3xTF32
    result must stay within a few times the FP32 FFMA error."""
    from gpu_util import normwise_err
    import oracle
    M, N, K = 256, 256, 2048
    A, B, _ = make_inputs(M, N, K, "uniform", seed=77)
    ref = oracle.sgemm(A, B)
    errs = {}
    for tc in (False, True):
        dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
        dC = torch.empty((M, N), device="cuda")
        sg.sgemm(dA, dB, dC, 1.0, 0.0, tensor_cores=tc)
        assert sg.status() == sg.OK
        errs[tc] = normwise_err(dC.cpu().numpy(), ref, A, B, K)
    # one-term TF32 would be ~2^-11 / sqrt(K) relative, about 1e-5 on this gate
    assert errs[True] <= 4 * errs[False] + 1e-9, errs
    assert errs[True] < 1e-7, errs


def test_tf32x3_nan_propagates():
    M, N, K = 140, 64, 64
    A, B, _ = make_inputs(M, N, K, "uniform", seed=3)
    A[7, 9] = np.nan
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), device="cuda")
    sg.sgemm(dA, dB, dC, 1.0, 0.0, tensor_cores=True)
    assert sg.status() == sg.OK
    C = dC.cpu().numpy()
    assert np.isnan(C[7]).all() and np.isfinite(np.delete(C, 7, axis=0)).all()


# ---------------------------------------------------------------- two-SM tensor-core tiles
# M >= 256 runs on clusters of two CTAs (tcgen05 cta_group::2), each pair a
# 256 x 256 tile: exactly one pair tile, a second pair tile whose odd CTA
# holds no rows (M = 257) or whose rows are all past M (M = 384), B halves
# partly or wholly past N, K tails, more tiles than co-resident pairs (the
# persistent loop), and M = 255 (still one-SM tiles) for contrast.
@pytest.mark.parametrize("mode", [sg.MODE_3XTF32, sg.MODE_TF32, sg.MODE_BF16])
@pytest.mark.parametrize("M,N,K", [(256, 256, 16), (257, 300, 100), (384, 129, 33), (512, 1, 40),
                                   (255, 260, 70), (2048, 2560, 64)])
def test_pair_tiles(mode, M, N, K):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M + 3 * N + 7 * K + mode, beta=-0.75)
    kid = {sg.MODE_3XTF32: TF, sg.MODE_TF32: sg.KERNEL_TF32, sg.MODE_BF16: sg.KERNEL_BF16}[mode]
    _, chosen = run_checked(sg, A, B, C0, 1.5, -0.75, tensor_cores=mode)
    assert chosen == kid


# ---------------------------------------------------------------- FFMA tile configurations
# Every configuration compiled into the library (the autotuner's choices),
# forced, on shapes with ragged edges, a divided tail and beta != 0.
@pytest.mark.parametrize("cfg", range(6))
@pytest.mark.parametrize("M,N,K", [(300, 260, 516), (1500, 1100, 700), (129, 1000, 77),
                                   (2300, 2352, 1001), (31, 3000, 2050)])
def test_every_ffma_config(cfg, M, N, K):
    assert len(sg.ffma_configs()) == 6
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + cfg, beta=0.5)
    ldb = (N + 3) // 4 * 4
    prev = sg.ffma_force_config(cfg)
    try:
        _, chosen = run_checked(sg, A, B, C0, 1.5, 0.5, lds=(K, ldb, N + 1))
        assert chosen == TMA
        Ai, Bi, Ci = make_inputs(M, N, min(K, 300), "int", seed=cfg, beta=-1.0)
        run_checked(sg, Ai, Bi, Ci, 2.0, -1.0, exact=True, lds=(min(K, 300), ldb, N))
    finally:
        sg.ffma_force_config(prev)


# The partial tiles of a divided tail are summed either by a separate kernel
# over all tail tiles at once (the default) or by the last unit to reach each
# tile, inside the tile kernel.
# Both add the same partials in the same order and apply the same epilogue,
# so the two must agree bit for bit, and each must pass the oracle gate.
# Covered: the 128x128 and 32x256 configurations, few and many partials per
# tile, beta != 0, a fused bias + activation, and C rows that are not
# 16-byte aligned (the scalar store path).
TAIL_SUM_CASES = [
    (1000, 1000, 1000, -1, 0.5, None, "none", 0),
    (31, 3000, 2050, 4, 1.0, None, "none", 0),
    (32, 1024, 4096, 4, -0.75, "bias", "silu", 0),
    (300, 260, 516, 0, 1.25, None, "relu", 1),
    (513, 384, 3000, 2, 0.0, "bias", "gelu", 1),
]


@pytest.mark.parametrize("M,N,K,cfg,beta,bias,act,ragged_c", TAIL_SUM_CASES)
def test_tail_sum_by_kernel_matches_last_arriver(M, N, K, cfg, beta, bias, act, ragged_c):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + N + K, beta=beta)
    bvec = synth.matrix(1, N, seed=5, stream=3, dist="normal")[0] if bias else None
    ldb = (N + 3) // 4 * 4
    lds = (K, ldb, N + 1 if ragged_c else ldb)
    prev_cfg = sg.ffma_force_config(cfg)
    outs = []
    try:
        plan = sg.ffma_tail_plan(M, N, K)
        assert plan["span"] > 0 and plan["tail_sum"] == 1, plan   # divided, summed by the kernel
        for mode in (0, 1):
            prev = sg.ffma_force_tail_sum(mode)
            try:
                _, chosen, C = run_checked(sg, A, B, C0, 1.5, beta, lds=lds, bias=bvec, act=act,
                                           return_c=True)
            finally:
                sg.ffma_force_tail_sum(prev)
            assert chosen == TMA
            outs.append(C)
    finally:
        sg.ffma_force_config(prev_cfg)
    assert np.array_equal(outs[0], outs[1]), "the two ways of summing the tail differ"


# ---------------------------------------------------------------- fused epilogue
# C = act(alpha*A@B + beta*C + bias[j]) on every kernel path: the TMA tile
# kernel (whole tiles and a divided tail), the plain-load kernel, the
# decode kernels (both outer-product tiles, the TMA and the direct-load
# kernel), C = act(beta*C + bias) without the product, and the tensor-core
# kernels on one-SM and two-SM tiles in all three arithmetics.
EPI_CASES = [  # (M, N, K, kernel, tensor_cores, ldb padding, lda padding)
    (300, 260, 516, TMA, False, 0, 0),        # 9 tiles, divided by work
    (1100, 700, 200, TMA, False, 0, 0),       # whole tiles
    (150, 130, 70, GEN, False, 3, 0),
    (16, 1000, 512, DEC, False, 0, 0),        # outer-product decode kernel, 16-row tile
    (4, 1000, 700, DEC, False, 0, 0),         # outer-product decode kernel, 8-row tile
    (4, 1000, 700, DEC, False, 0, 1),         # TMA decode kernel (A unaligned)
    (8, 999, 700, DEC, False, 3, 0),          # direct-load decode kernel (B unaligned)
    (256, 384, 200, sg.KERNEL_TF32X3, True, 0, 0),           # two-SM tensor-core tiles
    (256, 384, 200, sg.KERNEL_TF32, sg.MODE_TF32, 0, 0),
    (256, 384, 200, sg.KERNEL_BF16, sg.MODE_BF16, 0, 0),
    (200, 384, 200, sg.KERNEL_TF32X3, True, 0, 0),           # one-SM tensor-core tiles
    (200, 384, 200, sg.KERNEL_TF32, sg.MODE_TF32, 0, 0),
    (200, 384, 200, sg.KERNEL_BF16, sg.MODE_BF16, 0, 0),
]


@pytest.mark.parametrize("act", ["none", "relu", "gelu", "silu"])
@pytest.mark.parametrize("M,N,K,kern,tc,pad,apad", EPI_CASES)
def test_fused_epilogue(M, N, K, kern, tc, pad, apad, act):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + N + K, beta=0.5)
    bias = synth.matrix(1, N, seed=M + K, stream=3, dist="normal")[0] * 4
    lds = (K + apad, N + pad, N + 1) if (pad or apad) else (None, None, None)
    _, chosen = run_checked(sg, A, B, C0, 0.1, 0.5, tensor_cores=tc, bias=bias, act=act, lds=lds)
    assert chosen == kern


@pytest.mark.parametrize("act", ["relu", "gelu", "silu"])
def test_fused_epilogue_without_product(act):
    M, N, K = 77, 130, 40
    A, B, C0 = make_inputs(M, N, K, "normal", seed=5, beta=1.0)
    bias = synth.matrix(1, N, seed=6, stream=3, dist="normal")[0]
    for alpha, k in ((0.0, K), (1.0, 0)):
        run_checked(sg, A[:, :k], B[:k], C0, alpha, -0.75, bias=bias, act=act)


def test_fused_epilogue_integers_exact_and_nan():
    # small integers: alpha*A@B + beta*C + bias is exact in FP32, and ReLU keeps it exact
    A, B, C0 = make_inputs(300, 260, 516, "int", seed=8, beta=1.0)
    bias = synth.matrix(1, 260, seed=8, stream=3, dist="int")[0] * 16
    run_checked(sg, A, B, C0, 2.0, -1.0, bias=bias, act="relu", exact=True)
    run_checked(sg, A[:4], B, C0[:4], 2.0, -1.0, bias=bias, act="relu", exact=True)
    # a NaN in C reaches the output through ReLU (not clamped to 0)
    C1 = C0.copy()
    C1[5, 7] = np.nan
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C1))
    sg.sgemm(dA, dB, dC, 1.0, 1.0, bias=torch.from_numpy(bias).cuda(), activation="relu")
    assert sg.status() == sg.OK
    C = dC.cpu().numpy()
    assert np.isnan(C[5, 7]) and np.isfinite(np.delete(C.reshape(-1), 5 * 260 + 7)).all()


def test_fused_epilogue_rejects_bad_arguments():
    dA = torch.randn(64, 32, device="cuda")
    dB = torch.randn(32, 48, device="cuda")
    dC = torch.zeros(64, 48, device="cuda")
    L = sg.lib()
    args = (64, 48, 32, 1.0, dA.data_ptr(), 32, dB.data_ptr(), 48, 0.0, dC.data_ptr(), 48)
    assert L.sgemm_fused(*args, None, 4, 0, None) == sg.ERR_BAD_ARG          # activation
    assert L.sgemm_fused(*args, None, 1, 4, None) == sg.ERR_BAD_ARG          # mode
    assert L.sgemm_fused(*args, dC.data_ptr() + 4 * 48 * 10, 1, 0, None) == sg.ERR_ALIAS
    with pytest.raises(ValueError):
        sg.sgemm(dA, dB, dC, activation="tanh")
    with pytest.raises(TypeError):
        sg.sgemm(dA, dB, dC, bias=torch.zeros(47, device="cuda"))
    torch.cuda.synchronize()
    assert (dC == 0).all()


# ---------------------------------------------------------------- 1xTF32 (sgemm_tf32)
# The contract: A and B rounded to TF32 (nearest, ties away), then the FP32
# product -- checked against the oracle on rounded operands at the FP32 gate.
TF1 = sg.KERNEL_TF32


@pytest.mark.parametrize("M,N,K", [(17, 8, 8), (128, 256, 16), (129, 257, 40), (300, 520, 1000),
                                   (1000, 1000, 1000), (257, 300, 4097)])
def test_tf32_shapes(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M * 5 + N + K, beta=0.5)
    _, chosen = run_checked(sg, A, B, C0, 1.25, 0.5, tensor_cores=sg.MODE_TF32)
    assert chosen == TF1


def test_tf32_small_integers_exact_and_layouts():
    A, B, C0 = make_inputs(300, 200, 1000, "int", seed=6, beta=-2.0)
    run_checked(sg, A, B, C0, 3.0, -2.0, tensor_cores=sg.MODE_TF32, exact=True)
    A, B, C0 = make_inputs(70, 45, 33, "int", seed=13, beta=1.0)
    for lds, offsets in [((37, 47, 46), (1, 3, 1)), ((40, 48, 48), (0, 0, 0))]:
        run_checked(sg, A, B, C0, -1.0, 0.5, lds=lds, offsets=offsets,
                    tensor_cores=sg.MODE_TF32, exact=True)


def test_tf32_rounding_matches_the_oracle():
    """With B = I the product is round(A) exactly (and round(B) with A = I), so
    the GPU's TF32 rounding is compared with the oracle's element by element:
    random values, values just below / at / above a tie, negative ties."""
    import oracle
    n = 256
    rng = np.random.default_rng(11)
    A = rng.standard_normal((n, n)).astype(np.float32) * 3
    bits = A.view(np.uint32)
    bits[:64] = (bits[:64] & 0xffffe000) | 0x1000                # exact ties
    bits[64:96] = (bits[64:96] & 0xffffe000) | 0x0fff            # just below
    bits[96:128] = (bits[96:128] & 0xffffe000) | 0x1001          # just above
    eye = np.eye(n, dtype=np.float32)
    for X, Y, want in ((A, eye, oracle.round_tf32(A)), (eye, A, oracle.round_tf32(A))):
        dX, dY = torch.from_numpy(X).cuda(), torch.from_numpy(Y).cuda()
        dC = torch.empty((n, n), device="cuda")
        sg.sgemm_tf32(dX, dY, dC)
        assert sg.status() == sg.OK
        got = dC.cpu().numpy()
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, f"{bad.size} elements differ, first {got.flat[bad[0]]!r} vs {want.flat[bad[0]]!r}"


def test_tf32_is_one_term():
    """On uniform inputs (24 significant bits) the 1xTF32 result is within the
    FP32 gate of the rounded-operand product but visibly off the exact one."""
    from gpu_util import normwise_err
    import oracle
    M, N, K = 256, 256, 2048
    A, B, _ = make_inputs(M, N, K, "uniform", seed=78)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), device="cuda")
    sg.sgemm_tf32(dA, dB, dC)
    assert sg.status() == sg.OK
    got = dC.cpu().numpy()
    err_rounded = normwise_err(got, oracle.sgemm(A, B, inputs="tf32"), A, B, K)
    err_exact = normwise_err(got, oracle.sgemm(A, B), A, B, K)
    assert err_rounded <= GATE, err_rounded
    assert err_exact > 3 * GATE, err_exact


# ---------------------------------------------------------------- BF16 (sgemm_bf16)
# The contract: A and B rounded to BF16 (nearest, ties to even), then the FP32
# product -- checked against the oracle on rounded operands at the FP32 gate.
BF = sg.KERNEL_BF16


@pytest.mark.parametrize("M,N,K", [(17, 8, 8), (128, 256, 32), (129, 257, 40), (300, 520, 1000),
                                   (1000, 1000, 1000), (257, 300, 4097)])
def test_bf16_shapes(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M * 3 + N + K, beta=0.5)
    _, chosen = run_checked(sg, A, B, C0, 1.25, 0.5, tensor_cores=sg.MODE_BF16)
    assert chosen == BF


def test_bf16_small_integers_exact_and_layouts():
    A, B, C0 = make_inputs(300, 200, 1000, "int", seed=7, beta=-2.0)
    run_checked(sg, A, B, C0, 3.0, -2.0, tensor_cores=sg.MODE_BF16, exact=True)
    A, B, C0 = make_inputs(70, 45, 33, "int", seed=14, beta=1.0)
    for lds, offsets in [((37, 47, 46), (1, 3, 1)), ((40, 48, 48), (0, 0, 0))]:
        run_checked(sg, A, B, C0, -1.0, 0.5, lds=lds, offsets=offsets,
                    tensor_cores=sg.MODE_BF16, exact=True)


def test_bf16_rounding_matches_the_oracle():
    """B = I gives round(A) exactly (A = I gives round(B)): the GPU's BF16
    rounding against the oracle's, including ties in both directions."""
    import oracle
    n = 256
    rng = np.random.default_rng(12)
    A = rng.standard_normal((n, n)).astype(np.float32) * 3
    bits = A.view(np.uint32)
    bits[:64] = (bits[:64] & 0xffff0000) | 0x8000                # exact ties
    bits[64:96] = (bits[64:96] & 0xffff0000) | 0x7fff            # just below
    bits[96:128] = (bits[96:128] & 0xffff0000) | 0x8001          # just above
    eye = np.eye(n, dtype=np.float32)
    want = oracle.round_bf16(A)
    for X, Y in ((A, eye), (eye, A)):
        dX, dY = torch.from_numpy(X).cuda(), torch.from_numpy(Y).cuda()
        dC = torch.empty((n, n), device="cuda")
        sg.sgemm_bf16(dX, dY, dC)
        assert sg.status() == sg.OK
        got = dC.cpu().numpy()
        bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
        assert bad.size == 0, f"{bad.size} elements differ, first {got.flat[bad[0]]!r} vs {want.flat[bad[0]]!r}"


def test_bf16_is_bf16():
    """Within the FP32 gate of the product of BF16-rounded operands, and far
    from both the exact product and the TF32-rounded one."""
    from gpu_util import normwise_err
    import oracle
    M, N, K = 256, 256, 2048
    A, B, _ = make_inputs(M, N, K, "uniform", seed=79)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), device="cuda")
    sg.sgemm_bf16(dA, dB, dC)
    assert sg.status() == sg.OK
    got = dC.cpu().numpy()
    assert normwise_err(got, oracle.sgemm(A, B, inputs="bf16"), A, B, K) <= GATE
    assert normwise_err(got, oracle.sgemm(A, B), A, B, K) > 30 * GATE
    assert normwise_err(got, oracle.sgemm(A, B, inputs="tf32"), A, B, K) > 30 * GATE


# ---------------------------------------------------------------- large ragged shapes
# More tiles than resident blocks, ragged edges in M and N, K not a multiple of
# the 32-deep k-tile; every output compared.
@pytest.mark.parametrize("M,N,K,beta", [(2300, 2350, 700, 0.7), (2431, 2305, 1001, 0.0)])
def test_large_ragged_full_compare(M, N, K, beta):
    A, B, C0 = make_inputs(M, N, K, "uniform", seed=M + K, beta=beta)
    ldb = (N + 3) // 4 * 4        # B must be TMA-readable; N itself stays ragged
    _, chosen = run_checked(sg, A, B, C0, 1.5, beta, lds=(K, ldb, N))
    assert chosen == TMA


# Shapes whose tail (the tiles after the last full wave of resident blocks,
# all of them when they fill less than one wave) is divided by work into equal
# runs of K iterations; every output compared, and a second call is bitwise
# equal.
@pytest.mark.parametrize("M,N,K,beta,ldc_pad", [(1000, 1000, 1000, 0.0, 0), (1500, 1100, 700, -0.4, 5),
                                                (1001, 999, 513, 1.0, 3)])
def test_split_last_wave(M, N, K, beta, ldc_pad):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=M + N + K, beta=beta)
    ldb = (N + 3) // 4 * 4
    _, chosen = run_checked(sg, A, B, C0, 0.8, beta, lds=(K, ldb, N + ldc_pad))
    assert chosen == TMA
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = []
    for _ in range(2):
        dC = torch.from_numpy(C0).cuda()
        sg.sgemm(dA, dB, dC, 0.8, beta)
        assert sg.status() == sg.OK
        outs.append(dC.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


# Skinny products, 17 <= M <= 128 (the band between the decode kernel and
# full tiles: 32-row tiles, the tail divided by work so the few tiles fill the GPU);
# ragged M, N and K, every output compared.
SK_M = [17, 24, 31, 32, 33, 48, 63, 64, 65, 100, 127, 128]
SK_NK = [(257, 100), (3001, 1031), (14336, 4096)]


@pytest.mark.parametrize("N,K", SK_NK)
@pytest.mark.parametrize("M", SK_M)
def test_skinny_band(M, N, K):
    A, B, C0 = make_inputs(M, N, K, "normal", seed=31 * M + N + K, beta=0.5, sigma_b=0.02)
    ldb = (N + 3) // 4 * 4
    _, chosen = run_checked(sg, A, B, C0, 1.0, 0.5, lds=(K, ldb, N))
    # products of at most 2^21 multiply-adds take the one-launch plain-load kernel
    assert chosen == (GEN if M * N * K <= 1 << 21 else TMA)


@pytest.mark.parametrize("M", [17, 32, 64, 128])
def test_skinny_band_integers_exact(M):
    A, B, C0 = make_inputs(M, 14336, 4096, "int", seed=M, beta=-1.0)
    _, chosen = run_checked(sg, A, B, C0, 1.0, -1.0, exact=True)
    assert chosen == TMA


def test_large_small_integers_exact():
    A, B, C0 = make_inputs(2200, 2400, 300, "int", seed=9, beta=-1.0)
    _, chosen = run_checked(sg, A, B, C0, 2.0, -1.0, exact=True)
    assert chosen == TMA


def test_kernel_timing_hook():
    # the events bracket the tile kernel only: its time is below the calls'
    # time, one record per FFMA-path call, none for the decode path
    import oracle
    from gpu_util import normwise_err
    M = N = K = 1024
    A, B, C0 = make_inputs(M, N, K, "normal", seed=5)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.empty((M, N), device="cuda")
    dA16 = dA[:16].contiguous()
    dC16 = torch.empty((16, N), device="cuda")
    assert sg.lib().sgemm_kernel_timing(2) == sg.ERR_BAD_ARG
    assert sg.kernel_timing(True) == 0
    try:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            sg.sgemm(dA, dB, dC)
            sg.sgemm(dA16, dB, dC16)
        e1.record()
        torch.cuda.synchronize()
    finally:
        assert sg.kernel_timing(False) == 1
    total, n = sg.kernel_timing_result()
    assert n == 3
    assert 0.0 < total < e0.elapsed_time(e1)
    assert sg.status() == sg.OK
    ref = oracle.sgemm(A, B, alpha=1.0, beta=0.0)
    assert normwise_err(dC.cpu().numpy(), ref, A, B, K) <= GATE
    # stopped: later calls add nothing
    sg.sgemm(dA, dB, dC)
    torch.cuda.synchronize()
    assert sg.kernel_timing_result()[1] == 3
