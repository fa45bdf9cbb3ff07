"""Seeded synthetic matrices for the SGEMM workloads.

This module is the one piece that both sides of the parity check share: the
fp64 CPU oracle and the CUDA library receive bit-identical float32 arrays made
here.  It holds no GEMM arithmetic, only a counter-based random generator and
the three value distributions the workloads use.

Generator (counter-based SplitMix64, S. Vigna's published mixing function):

    key      = mix64((seed << 8) | stream)
    raw(i)   = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)        (mod 2**64)
    mix64(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)

Element ``i`` of a matrix is its row-major index ``r * cols + c`` (independent
of the leading dimension, so padding never changes the values).  Streams keep
A, B and C apart: A=0, B=1, C=2.

Distributions (all values are produced in fp64 and rounded once to float32):

* ``uniform``  [-1, 1):  (raw >> 40) * 2**-23 - 1   -- 24 random bits, exact in fp32
* ``normal``   N(mean, sigma): Box-Muller on raw(2i), raw(2i+1):
               u1 = ((raw(2i) >> 11) + 1) * 2**-53   in (0, 1]
               u2 =  (raw(2i+1) >> 11)    * 2**-53   in [0, 1)
               z  = sqrt(-2 ln u1) * cos(2 pi u2)
* ``int``      small integers in [-4, 4]: floor(u * 9) - 4, u = (raw >> 11) * 2**-53

The workloads (shapes, seeds, distributions) are listed in ``WORKLOADS``.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

STREAM_A, STREAM_B, STREAM_C = 0, 1, 2

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser, in place on a uint64 array (wrapping arithmetic)."""
    t = np.empty_like(z)
    np.right_shift(z, np.uint64(30), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, _M1, out=z)
    np.right_shift(z, np.uint64(27), out=t)
    np.bitwise_xor(z, t, out=z)
    np.multiply(z, _M2, out=z)
    np.right_shift(z, np.uint64(31), out=t)
    np.bitwise_xor(z, t, out=z)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    if not (0 <= stream < 256) or seed < 0:
        raise ValueError("seed must be >= 0 and stream in [0, 256)")
    base = np.array([((seed << 8) | stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Outputs ``raw(start) .. raw(start + count - 1)`` of one stream."""
    key = _key(seed, stream)
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        np.multiply(z, _GOLDEN, out=z)
        np.add(z, key, out=z)
        return _mix64(z)


def _fill_chunk(flat: np.ndarray, s: int, c: int, seed: int, stream: int, dist: str,
                mean: float, sigma: float) -> None:
    if dist == "uniform":
        r = raw_u64(seed, stream, s, c)
        v = (r >> np.uint64(40)).astype(np.float64)
        v *= 2.0**-23
        v -= 1.0
    elif dist == "int":
        r = raw_u64(seed, stream, s, c)
        v = (r >> np.uint64(11)).astype(np.float64)
        v *= 2.0**-53 * 9.0
        np.floor(v, out=v)
        v -= 4.0
    elif dist == "normal":
        r = raw_u64(seed, stream, 2 * s, 2 * c)
        u1 = (r[0::2] >> np.uint64(11)).astype(np.float64)
        u1 += 1.0
        u1 *= 2.0**-53
        u2 = (r[1::2] >> np.uint64(11)).astype(np.float64)
        u2 *= 2.0**-53 * 2.0 * np.pi
        np.log(u1, out=u1)
        u1 *= -2.0
        np.sqrt(u1, out=u1)
        np.cos(u2, out=u2)
        v = u1 * u2
        v *= sigma
        v += mean
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    flat[s:s + c] = v


def _fill(out: np.ndarray, seed: int, stream: int, dist: str, mean: float, sigma: float) -> None:
    flat = out.reshape(-1)
    n = flat.size
    starts = list(range(0, n, _CHUNK))
    work = [(s, min(_CHUNK, n - s)) for s in starts]
    if len(work) == 1:
        _fill_chunk(flat, *work[0], seed, stream, dist, mean, sigma)
        return
    workers = min(len(work), os.cpu_count() or 1, 16)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda w: _fill_chunk(flat, w[0], w[1], seed, stream, dist, mean, sigma), work))


def matrix(rows: int, cols: int, *, seed: int, stream: int, dist: str = "uniform",
           mean: float = 0.0, sigma: float = 1.0, ld: int | None = None,
           pad_value: float = float("nan")) -> np.ndarray:
    """A ``rows x cols`` float32 matrix, row-major.

    With ``ld > cols`` the result is a view into a ``rows x ld`` buffer whose
    gap columns hold ``pad_value`` (NaN by default, so a kernel that reads the
    gap poisons its output).  ``ld`` defaults to ``cols``.
    """
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld must be >= cols")
    vals = np.empty((rows, cols), dtype=np.float32)
    if vals.size:
        _fill(vals, seed, stream, dist, mean, sigma)
    if ld == cols:
        return vals
    buf = np.full((rows, ld), pad_value, dtype=np.float32)
    buf[:, :cols] = vals
    return buf[:, :cols]


# The workloads the library is measured and checked on.  Shapes are
# (M, N, K): A is M x K, B is K x N, C is M x N.
WORKLOADS = {
    "sgemm_128": dict(M=128, N=128, K=128, alpha=1.0, beta=0.0, seed=0,
                      a=("uniform", 0.0, 1.0), b=("uniform", 0.0, 1.0), c=None),
    "sgemm_128_int": dict(M=128, N=128, K=128, alpha=1.0, beta=0.0, seed=0,
                          a=("int", 0.0, 1.0), b=("int", 0.0, 1.0), c=None),
    "sgemm_4092": dict(M=4092, N=4092, K=4092, alpha=1.0, beta=0.5, seed=1,
                       a=("uniform", 0.0, 1.0), b=("uniform", 0.0, 1.0),
                       c=("uniform", 0.0, 1.0)),
    "sgemm_8192": dict(M=8192, N=8192, K=8192, alpha=1.0, beta=0.0, seed=2,
                       a=("normal", 0.0, 1.0), b=("normal", 0.0, 1.0), c=None),
    "decode_m1": dict(M=1, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                      a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "decode_m4": dict(M=4, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                      a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "decode_m16": dict(M=16, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                       a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    # skinny products on the decode shapes' N, K and B (the band between
    # the decode kernel and full tiles)
    "skinny_m32": dict(M=32, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                       a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "skinny_m64": dict(M=64, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                       a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "skinny_m128": dict(M=128, N=14336, K=4096, alpha=1.0, beta=0.0, seed=3,
                        a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "prefill_qkv": dict(M=8192, N=12288, K=4096, alpha=1.0, beta=0.0, seed=4,
                        a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "prefill_up": dict(M=8192, N=14336, K=4096, alpha=1.0, beta=0.0, seed=4,
                       a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
    "prefill_down": dict(M=8192, N=4096, K=14336, alpha=1.0, beta=0.0, seed=4,
                         a=("normal", 0.0, 1.0), b=("normal", 0.0, 0.02), c=None),
}


def workload_inputs(name: str):
    """(A, B, C0-or-None, spec) for one named workload."""
    w = WORKLOADS[name]
    M, N, K, seed = w["M"], w["N"], w["K"], w["seed"]
    da, ma, sa = w["a"]
    db, mb, sb = w["b"]
    A = matrix(M, K, seed=seed, stream=STREAM_A, dist=da, mean=ma, sigma=sa)
    B = matrix(K, N, seed=seed, stream=STREAM_B, dist=db, mean=mb, sigma=sb)
    C = None
    if w["c"] is not None:
        dc, mc, sc = w["c"]
        C = matrix(M, N, seed=seed, stream=STREAM_C, dist=dc, mean=mc, sigma=sc)
    return A, B, C, w
