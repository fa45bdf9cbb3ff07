"""Host-side logic of bench.py (no GPU): the acceptance gate it reports, the
row/column samples of its parity checks, and the source hash that decides
whether a recorded ncu traffic figure still applies."""

import numpy as np
import pytest

import bench
import oracle
import synth


def test_gate_is_verbatim_without_beta():
    A = np.full((2, 3), 2.0, np.float32)
    B = np.full((3, 2), 0.5, np.float32)
    ref = np.full((2, 2), 3.0)
    got = ref.copy()                              # float64, so the offset is exact
    got[1, 1] += 3 * 2.0 * 0.5 * 1e-6          # exactly the gate: K * max|A| * max|B| * 1e-6
    assert bench.gate_err(got, ref, A, B, 3, 1.0, 0.0, None) == pytest.approx(1e-6)
    got[1, 1] += 1e-6
    assert bench.gate_err(got, ref, A, B, 3, 1.0, 0.0, None) > 1e-6


def test_gate_allows_the_rounding_of_beta_c_per_element():
    A = np.ones((1, 1), np.float32)
    B = np.ones((1, 1), np.float32) * 1e-3
    C0 = np.array([[1e6, 1.0]], np.float32)
    ref = np.array([[1e6, 1.0]], np.float64)
    # one ulp of 1e6 (0.0625) is far above the product gate (1e-9) but within
    # 2^-22 * (|beta*C0| + |C_ref|) of that element ...
    got = np.array([[1e6 + 0.0625, 1.0]], np.float32)
    assert bench.gate_err(got, ref, A, B, 1, 1.0, 1.0, C0) <= 1e-6
    # ... while the same absolute error on the small element is not
    got = np.array([[1e6, 1.0625]], np.float32)
    assert bench.gate_err(got, ref, A, B, 1, 1.0, 1.0, C0) > 1e-6


def test_nan_fails_the_gate():
    A = B = np.ones((2, 2), np.float32)
    got = np.array([[np.nan, 2.0], [2.0, 2.0]], np.float32)
    assert bench.gate_err(got, np.full((2, 2), 2.0), A, B, 2, 1.0, 0.0, None) == float("inf")


def test_sample_index_hits_every_tile_band():
    for n in (1, 60, 61, 62, 4092, 14336):
        idx = bench.sample_index(n)
        assert idx[0] == 0 and idx[-1] == n - 1
        assert np.all(np.diff(idx) <= 61)           # every 32- or 128-wide band contains one


@pytest.mark.parametrize("M,N,K", [(70, 90, 33), (300, 200, 50)])
def test_parity_check_full_and_cross_sample(M, N, K):
    A = synth.matrix(M, K, seed=5, stream=0, dist="uniform")
    B = synth.matrix(K, N, seed=5, stream=1, dist="uniform")
    C0 = synth.matrix(M, N, seed=5, stream=2, dist="uniform")
    good = oracle.sgemm(A, B, C0, alpha=1.0, beta=0.5)
    for full in (1e12, 0.0):                         # every element, then the row/column cross
        assert bench.parity_check(A, B, C0, 1.0, 0.5, good, full_below_flop=full)["pass"]
        bad = good.copy()
        bad[M - 1, 7] += 1.0                          # a sampled row (the last one)
        r = bench.parity_check(A, B, C0, 1.0, 0.5, bad, full_below_flop=full)
        assert not r["pass"] and r["normwise_err"] > 1e-6


def test_source_hash_ignores_comments_only():
    code = 'int f(int x) { return x + 1; } // add\n/* note */ const char *s = "a // b";\n'
    same = 'int f(int x) {\n  return x + 1;   // one more\n}\nconst char *s = "a // b";\n'
    other = 'int f(int x) { return x + 2; }\nconst char *s = "a // b";\n'
    strings = 'int f(int x) { return x + 1; }\nconst char *s = "a // c";\n'
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(other)
    assert bench._code_only(code) != bench._code_only(strings)


PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2000.0, "_source": "measured"}


def test_roofline_ffma_uses_the_tile_kernel_time_when_given():
    import dense_fp32_matrix_row_gb300 as sg
    M = N = K = 1000
    flops = 2 * M * N * K
    b, ach, peak, unit, _ = bench.roofline_for(sg.KERNEL_FFMA_TMA, M, N, K, 0.5, 0.2, 0.1, 100, PEAKS)
    assert (b, unit) == ("alu", "TFLOP/s")
    assert peak == pytest.approx(100 * 128 * 2 * 2000e6 / 1e12)
    assert ach == pytest.approx(flops / 0.1e-3 / 1e12)              # the kernel's own 0.1 ms
    _, ach2, _, _, _ = bench.roofline_for(sg.KERNEL_FFMA_TMA, M, N, K, 0.5, 0.2, None, 100, PEAKS)
    assert ach2 == pytest.approx(flops / 0.2e-3 / 1e12)             # else the whole call


def test_roofline_tensor_and_decode_bounds():
    import dense_fp32_matrix_row_gb300 as sg
    M = N = K = 1000
    flops = 2 * M * N * K
    b, ach, peak, _, _ = bench.roofline_for(sg.KERNEL_TF32X3, M, N, K, 0.0, 0.1, None, 100, PEAKS)
    assert b == "tensor" and ach == pytest.approx(3 * flops / 0.1e-3 / 1e12)
    assert peak == pytest.approx(1900.0 * 1.1 / 2.25)
    b, ach, peak, _, _ = bench.roofline_for(sg.KERNEL_BF16, M, N, K, 0.0, 0.1, None, 100, PEAKS)
    assert b == "tensor" and ach == pytest.approx(flops / 0.1e-3 / 1e12) and peak == 1900.0
    # decode: bytes of A, B and C (read too when beta != 0) against the copy bandwidth
    b, ach, peak, unit, _ = bench.roofline_for(sg.KERNEL_DECODE, 16, 14336, 4096, 1.0, 0.05, None, 100,
                                              PEAKS)
    assert (b, unit, peak) == ("hbm", "GB/s", 6800.0)
    nbytes = 4 * (16 * 4096 + 4096 * 14336 + 2 * 16 * 14336)
    assert ach == pytest.approx(nbytes / 0.05e-3 / 1e9)
