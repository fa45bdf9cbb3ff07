"""The seeded generator against a scalar restatement of its published definition."""

import math

import numpy as np
import pytest

import synth

_M = (1 << 64) - 1


def _mix(z):
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _M
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _M
    return z ^ (z >> 31)


def _scalar(seed, stream, n, dist, sigma=1.0):
    key = _mix((seed << 8) | stream)
    raw = lambda i: _mix((key + (i + 1) * 0x9E3779B97F4A7C15) & _M)
    out = []
    for i in range(n):
        if dist == "uniform":
            out.append((raw(i) >> 40) * 2.0**-23 - 1.0)
        elif dist == "int":
            out.append(math.floor((raw(i) >> 11) * 2.0**-53 * 9.0) - 4.0)
        else:
            u1 = ((raw(2 * i) >> 11) + 1) * 2.0**-53
            u2 = (raw(2 * i + 1) >> 11) * 2.0**-53
            out.append(sigma * math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2))
    return np.array(out, dtype=np.float32)


@pytest.mark.parametrize("dist,sigma", [("uniform", 1.0), ("int", 1.0), ("normal", 0.02)])
def test_matches_scalar_definition(dist, sigma):
    # 3 x 1_400_000 spans two generator chunks, so the threaded path is covered
    got = synth.matrix(3, 1_400_000, seed=5, stream=1, dist=dist, sigma=sigma).reshape(-1)
    idx = np.r_[0:2000, (1 << 20) - 5:(1 << 20) + 5, got.size - 10:got.size]
    want_head = _scalar(5, 1, 2000, dist, sigma)
    assert np.array_equal(got[:2000], want_head)
    # spot-check elements far into the stream through the raw-index formula
    for i in map(int, idx[2000:]):
        key = _mix((5 << 8) | 1)
        if dist == "normal":
            r0 = _mix((key + (2 * i + 1) * 0x9E3779B97F4A7C15) & _M)
            r1 = _mix((key + (2 * i + 2) * 0x9E3779B97F4A7C15) & _M)
            u1 = ((r0 >> 11) + 1) * 2.0**-53
            u2 = (r1 >> 11) * 2.0**-53
            v = np.float32(sigma * math.sqrt(-2 * math.log(u1)) * math.cos(2 * math.pi * u2))
        else:
            r = _mix((key + (i + 1) * 0x9E3779B97F4A7C15) & _M)
            v = np.float32((r >> 40) * 2.0**-23 - 1.0 if dist == "uniform"
                           else math.floor((r >> 11) * 2.0**-53 * 9.0) - 4.0)
        assert got[i] == v


def test_ranges_and_padding():
    u = synth.matrix(50, 70, seed=1, stream=0, dist="uniform")
    assert u.min() >= -1.0 and u.max() < 1.0
    k = synth.matrix(50, 70, seed=1, stream=0, dist="int")
    assert set(np.unique(k)) <= set(range(-4, 5)) and len(np.unique(k)) == 9
    p = synth.matrix(5, 6, seed=1, stream=0, ld=9)
    assert p.shape == (5, 6) and p.strides == (36, 4)
    assert np.isnan(p.base[:, 6:]).all()
    assert np.array_equal(p, synth.matrix(5, 6, seed=1, stream=0))
    assert not np.array_equal(synth.matrix(4, 4, seed=1, stream=0), synth.matrix(4, 4, seed=1, stream=1))
