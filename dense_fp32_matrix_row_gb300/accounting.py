"""Work, traffic and roofline arithmetic for the SGEMM path (host logic only).

The counting rules follow the pages' own first-principles estimates:

* FLOPs: 2*M*N*K multiply-add work (an FMA counts as two), plus M*N for the
  alpha/beta epilogue when it is counted ("GPU GEMM 优化完全拆解（一）", section
  "什么是 GEMM"; "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section
  "1. Kernel 1", first-principles estimate).  Benchmarks report 2*M*N*K.
* Minimum DRAM traffic: read A, B (and C when beta != 0) once, write C once
  (same section of "CUDA 矩阵乘法优化"; "GPU GEMM 优化完全拆解（一）", section
  "理论下限").
* Shared-memory tiling moves 4*M*N*K*(1/BM + 1/BN) bytes of A and B
  ("GPU GEMM 优化完全拆解（一）", section "收益：全局内存流量降了一个量级").
* Per-output loads of a BMxBN block tile with TMxTN thread tiles: K*(1/BM+1/BN)
  global and K*(TM+TN)/(TM*TN) shared ("CUDA 矩阵乘法优化", sections 3, 5, 6).
* Arithmetic intensity = FLOPs / DRAM bytes; a TILE x TILE shared tile gives
  TILE/4 FLOP/B ("GPU 基础原理", sections 2 and 4.7).
* Occupancy: the minimum over the thread, register (per-warp allocation
  granularity) and shared-memory ceilings ("GPU GEMM 优化完全拆解（一）",
  section "占用率的定义与三个资源天花板").
"""

from __future__ import annotations

import math
from dataclasses import dataclass

F32 = 4  # bytes per element


def gemm_flops(M: int, N: int, K: int, epilogue: bool = False) -> int:
    """2*M*N*K, plus M*N when the alpha/beta epilogue is counted."""
    return 2 * M * N * K + (M * N if epilogue else 0)


def min_traffic_bytes(M: int, N: int, K: int, beta_nonzero: bool = True) -> int:
    """Bytes any implementation must move: read A, B (and C if beta != 0), write C."""
    return F32 * (M * K + K * N + M * N * (2 if beta_nonzero else 1))


def naive_traffic_bytes(M: int, N: int, K: int) -> int:
    """One thread per output, no reuse: each reads a row of A, a column of B
    and its C element, 2K+1 floats."""
    return F32 * M * N * (2 * K + 1)


def tiled_ab_traffic_bytes(M: int, N: int, K: int, BM: int, BN: int) -> float:
    """A and B bytes moved by BMxBN block tiles sweeping K: 4*M*N*K*(1/BM + 1/BN)."""
    return F32 * M * N * K * (1.0 / BM + 1.0 / BN)


def loads_per_output(K: int, BM: int, BN: int, TM: int = 1, TN: int = 1):
    """(global, shared) float loads per output element for block tile BMxBN and
    thread tile TMxTN."""
    return K * (1.0 / BM + 1.0 / BN), K * (TM + TN) / (TM * TN)


def arithmetic_intensity(flops: float, nbytes: float) -> float:
    return flops / nbytes


def tile_intensity(tile: int) -> float:
    """FLOP/B of one TILE x TILE output tile computed from two TILE x TILE input
    tiles: 2*T^3 / (8*T^2)."""
    return (2 * tile**3) / (2 * F32 * tile**2)


def tile_grid(extent: int, tile: int):
    """(number of tiles, valid elements in the last tile) along one dimension."""
    n = math.ceil(extent / tile)
    return n, extent - (n - 1) * tile if n else 0


@dataclass(frozen=True)
class SMLimits:
    max_threads: int
    max_warps: int
    registers: int
    reg_granularity: int   # registers allocated per warp come in multiples of this
    smem_bytes: int
    smem_per_block_overhead: int = 0
    max_blocks: int = 32


A6000 = SMLimits(max_threads=1536, max_warps=48, registers=65536, reg_granularity=256,
                 smem_bytes=100 * 1024, smem_per_block_overhead=1024, max_blocks=16)
# GB300 (sm_103): 2048 threads, 64 warps, 64K registers, 228 KB shared per SM
# (227 KB usable per block), 1 KB reserved per block.
GB300 = SMLimits(max_threads=2048, max_warps=64, registers=65536, reg_granularity=256,
                 smem_bytes=228 * 1024, smem_per_block_overhead=1024, max_blocks=32)


def blocks_per_sm(threads: int, regs_per_thread: int, smem_bytes: int, lim: SMLimits) -> int:
    """Resident blocks per SM: the smallest of the three resource ceilings."""
    warps = math.ceil(threads / 32)
    by_threads = lim.max_threads // threads
    per_warp = math.ceil(regs_per_thread * 32 / lim.reg_granularity) * lim.reg_granularity
    by_regs = lim.registers // (per_warp * warps) if regs_per_thread else lim.max_blocks
    need = smem_bytes + lim.smem_per_block_overhead
    by_smem = lim.smem_bytes // need if need else lim.max_blocks
    return max(0, min(by_threads, by_regs, by_smem, lim.max_blocks))


def occupancy(threads: int, regs_per_thread: int, smem_bytes: int, lim: SMLimits) -> float:
    b = blocks_per_sm(threads, regs_per_thread, smem_bytes, lim)
    return b * math.ceil(threads / 32) / lim.max_warps


# ---- GB300 roofline denominators -------------------------------------------------

GB300_SMS = 152
FP32_LANES_PER_SM = 128      # 4 sub-partitions x 32 FP32 lanes
GB300_MAX_SM_MHZ = 2070.0


def ffma_peak_tflops(sms: int = GB300_SMS, sm_mhz: float = GB300_MAX_SM_MHZ,
                     lanes: int = FP32_LANES_PER_SM) -> float:
    """FP32 FFMA peak: SMs x lanes x 2 FLOP x clock."""
    return sms * lanes * 2 * sm_mhz * 1e6 / 1e12


# Nominal dense tensor rates (PFLOP/s) used only to scale a measured bf16 peak
# to another operand type.
NOMINAL_DENSE_PFLOPS = {"bf16": 2.25, "fp8": 4.5, "fp4": 13.5, "tf32": 1.1}


def tf32_peak_from_bf16(bf16_tflops: float) -> float:
    """Measured bf16 tensor peak scaled by the nominal tf32/bf16 ratio."""
    return bf16_tflops * NOMINAL_DENSE_PFLOPS["tf32"] / NOMINAL_DENSE_PFLOPS["bf16"]
