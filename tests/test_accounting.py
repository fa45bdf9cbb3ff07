"""Host accounting against the worked numbers printed on the pages (tests/golden)."""

import json
import os

import pytest

from dense_fp32_matrix_row_gb300 import accounting as acc

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
FIG = {f["name"]: f for f in GOLDEN["figures"]}
N = 4092


def close(value, fig):
    return abs(value - fig["printed"]) <= fig.get("tolerance", 1e-12)


def test_flops_4092():
    assert close(acc.gemm_flops(N, N, N, epilogue=True), FIG["flops_4092_with_epilogue"])
    assert acc.gemm_flops(N, N, N, epilogue=True) == FIG["flops_4092_misprint"]["exact"]
    # the benchmark counts the multiply-add work only
    assert acc.gemm_flops(N, N, N) == 2 * N**3


def test_min_traffic_4092():
    assert close(3 * N * N * 4, FIG["min_read_bytes_4092"])
    assert close(N * N * 4, FIG["min_write_bytes_4092"])
    assert close(acc.min_traffic_bytes(N, N, N, beta_nonzero=True), FIG["min_traffic_bytes_4092"])
    assert acc.min_traffic_bytes(N, N, N, beta_nonzero=False) == 3 * N * N * 4


def test_a6000_first_principles_times():
    flops = acc.gemm_flops(N, N, N, epilogue=True)
    t_c = flops / (FIG["a6000_compute_ms"]["args"]["peak_tflops"] * 1e12) * 1e3
    t_m = acc.min_traffic_bytes(N, N, N) / (FIG["a6000_memory_ms"]["args"]["bandwidth_gbs"] * 1e9) * 1e3
    assert close(t_c, FIG["a6000_compute_ms"])
    assert close(t_m, FIG["a6000_memory_ms"])
    assert close(t_c / t_m, FIG["compute_over_memory_ratio"])


def test_naive_and_tiled_traffic():
    assert close(acc.naive_traffic_bytes(N, N, N), FIG["naive_traffic_bytes_4092"])
    a = FIG["tiled32_traffic_bytes_4092"]["args"]
    assert close(acc.tiled_ab_traffic_bytes(N, N, N, a["BM"], a["BN"]), FIG["tiled32_traffic_bytes_4092"])


def test_tile_grids():
    assert list(acc.tile_grid(N, 32)) == FIG["grid_4092_by_32"]["printed"]
    assert [acc.tile_grid(65, 32)[0]] * 2 == FIG["grid_65_by_32"]["printed"]
    assert acc.tile_grid(0, 32) == (0, 0)


def test_arithmetic_intensity():
    n = 1000
    assert acc.arithmetic_intensity(2 * n, 8 * n) == FIG["ai_one_output_per_thread"]["printed"]
    assert acc.arithmetic_intensity(8 * n, 16 * n) == FIG["ai_2x2_per_thread"]["printed"]
    assert acc.tile_intensity(32) == FIG["ai_tile_32"]["printed"]
    assert acc.tile_intensity(64) == FIG["ai_tile_64"]["printed"]
    a = FIG["a100_ridge"]["args"]
    assert close(a["peak_tflops"] / a["bandwidth_tbs"], FIG["a100_ridge"])


@pytest.mark.parametrize("name", ["per_output_loads_kernel3", "per_output_loads_kernel4",
                                  "per_output_loads_kernel5"])
def test_per_output_loads(name):
    f = FIG[name]
    a = f["args"]
    K = 4096
    g, s = acc.loads_per_output(K, a["BM"], a["BN"], a["TM"], a["TN"])
    want = [c * K for c in f["per_K"]]
    assert g == pytest.approx(want[0]) and s == pytest.approx(want[1])


def test_occupancy_worked_example():
    f = FIG["a6000_kernel3_occupancy"]
    a = f["args"]
    lim = acc.A6000
    assert lim.smem_bytes // (a["smem"] + lim.smem_per_block_overhead) == f["printed"]["blocks_by_smem"]
    assert acc.blocks_per_sm(a["threads"], a["regs"], a["smem"], lim) == f["printed"]["blocks"]
    assert acc.occupancy(a["threads"], a["regs"], a["smem"], lim) == pytest.approx(f["printed"]["occupancy"], abs=0.01)


def test_gb300_ffma_peak():
    # 152 SMs x 128 lanes x 2 FLOP x 2070 MHz
    assert acc.ffma_peak_tflops() == pytest.approx(80.55, abs=0.01)
    assert acc.tf32_peak_from_bf16(2250.0) == pytest.approx(1100.0)
