"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
AssertionError when the handle's results contradict a fact that holds
independently of how the oracle is written:

* exact integer arithmetic (numpy int64) on small-integer matrices,
* exact rational arithmetic (``fractions.Fraction``) on tiny float inputs,
* closed forms: identity, permutation and rank-1 operands,
* the transpose identity (A@B)^T = B^T @ A^T,
* Freivalds' randomised check against numpy's fp64 matrix-vector products,
* the alpha/beta conventions (beta == 0 never reads C0; alpha == 0 never reads A, B),
* leading-dimension gaps filled with NaN canaries are never read.

``ALL_PINS`` lists them; ``tests/test_oracle_mutants.py`` plants mistakes in
copies of the oracle and checks that at least one pin fails for each.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

import synth


def _rng(seed):
    return np.random.default_rng(seed)


def pin_small_int_exact(orc):
    """Small integers in [-4, 4]: every partial sum is an integer below 2**24,
    so the float result is exact and must equal int64 arithmetic bit for bit."""
    for (M, N, K, seed) in [(37, 29, 53, 11), (128, 128, 128, 0), (5, 1, 300, 7), (1, 67, 2, 9)]:
        A = synth.matrix(M, K, seed=seed, stream=0, dist="int")
        B = synth.matrix(K, N, seed=seed, stream=1, dist="int")
        C0 = synth.matrix(M, N, seed=seed, stream=2, dist="int")
        exact = A.astype(np.int64) @ B.astype(np.int64)
        got = orc.sgemm(A, B)
        assert np.array_equal(got, exact.astype(np.float32)), "int A@B not exact"
        got = orc.sgemm(A, B, C0, alpha=2.0, beta=-3.0)
        want = 2 * exact - 3 * C0.astype(np.int64)
        assert np.array_equal(got, want.astype(np.float32)), "2*A@B - 3*C0 not exact"


def _frac(x):
    return Fraction(float(x))


def pin_exact_rational(orc):
    """Tiny float inputs against exact rational arithmetic: the oracle must
    agree with the exactly rounded value to within one float ulp."""
    for (M, N, K, alpha, beta, seed) in [(2, 3, 64, 0.75, -1.5, 21),
                                         (3, 2, 9, 1.0, 0.0, 22),
                                         (1, 4, 1, -2.5, 0.25, 23)]:
        A = synth.matrix(M, K, seed=seed, stream=0, dist="normal")
        B = synth.matrix(K, N, seed=seed, stream=1, dist="normal")
        C0 = synth.matrix(M, N, seed=seed, stream=2, dist="normal")
        got = orc.sgemm(A, B, C0 if beta != 0 else None, alpha=alpha, beta=beta)
        for i in range(M):
            for j in range(N):
                s = sum((_frac(A[i, k]) * _frac(B[k, j]) for k in range(K)), Fraction(0))
                ex = Fraction(alpha) * s
                if beta != 0:
                    ex += Fraction(beta) * _frac(C0[i, j])
                want = np.float32(float(ex))
                ulp = np.spacing(np.abs(want))
                assert abs(_frac(got[i, j]) - ex) <= Fraction(float(ulp)), \
                    f"element ({i},{j}) off the exact value by more than one ulp"


def pin_identity(orc):
    """A = I gives C = B and B = I gives C = A, bit for bit."""
    K = 37
    eye = np.eye(K, dtype=np.float32)
    B = synth.matrix(K, 23, seed=31, stream=1, dist="uniform")
    assert np.array_equal(orc.sgemm(eye, B), B), "I @ B != B"
    A = synth.matrix(19, K, seed=31, stream=0, dist="uniform")
    assert np.array_equal(orc.sgemm(A, eye), A), "A @ I != A"


def pin_permutation(orc):
    """A = P (row permutation) gives C = B[p]; B = P gives C = A[:, q] with
    q the inverse permutation.  A transposed operand fails this (P^T != P)."""
    rng = _rng(41)
    K = 45
    p = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), p] = 1.0
    B = synth.matrix(K, 31, seed=41, stream=1, dist="normal")
    assert np.array_equal(orc.sgemm(P, B), B[p]), "P @ B != B[p]"
    A = synth.matrix(13, K, seed=41, stream=0, dist="normal")
    q = np.argsort(p)
    assert np.array_equal(orc.sgemm(A, P), A[:, q]), "A @ P != A[:, p^-1]"


def pin_rank1(orc):
    """A[i,k] = u_i and B[k,j] = v_j give C[i,j] = K*u_i*v_j exactly (small
    integers), so every k must be counted exactly once."""
    for (M, N, K) in [(7, 9, 33), (16, 5, 1), (3, 3, 1000)]:
        u = (np.arange(M, dtype=np.float32) % 5) - 2
        v = (np.arange(N, dtype=np.float32) % 7) - 3
        A = np.repeat(u[:, None], K, axis=1).astype(np.float32)
        B = np.repeat(v[None, :], K, axis=0).astype(np.float32)
        want = (K * np.outer(u.astype(np.int64), v.astype(np.int64))).astype(np.float32)
        assert np.array_equal(orc.sgemm(A, B), want), f"rank-1 closed form fails at K={K}"


def pin_transpose(orc):
    """(alpha*A@B + beta*C0)^T = alpha*B^T@A^T + beta*C0^T, bit for bit (the
    same products are summed in the same k order)."""
    M, N, K = 21, 34, 17
    A = synth.matrix(M, K, seed=51, stream=0, dist="normal")
    B = synth.matrix(K, N, seed=51, stream=1, dist="normal")
    C0 = synth.matrix(M, N, seed=51, stream=2, dist="normal")
    C = orc.sgemm(A, B, C0, alpha=1.5, beta=-0.75)
    Ct = orc.sgemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                   np.ascontiguousarray(C0.T), alpha=1.5, beta=-0.75)
    assert np.array_equal(C, Ct.T), "transpose identity fails"


def pin_freivalds(orc):
    """C x = alpha*A(B x) + beta*C0 x for random sign vectors x, in fp64 numpy."""
    M, N, K = 67, 45, 129
    alpha, beta = 1.25, -0.5
    A = synth.matrix(M, K, seed=61, stream=0, dist="normal")
    B = synth.matrix(K, N, seed=61, stream=1, dist="normal")
    C0 = synth.matrix(M, N, seed=61, stream=2, dist="normal")
    C = orc.sgemm(A, B, C0, alpha=alpha, beta=beta).astype(np.float64)
    rng = _rng(61)
    scale = K * np.abs(A).max() * np.abs(B).max()
    for _ in range(3):
        x = rng.choice([-1.0, 1.0], size=N)
        lhs = C @ x
        rhs = alpha * (A.astype(np.float64) @ (B.astype(np.float64) @ x)) \
            + beta * (C0.astype(np.float64) @ x)
        err = np.abs(lhs - rhs).max() / (N * scale)
        assert err < 1e-6, f"Freivalds check off by {err:.3g}"


def pin_alpha_beta(orc):
    """alpha/beta conventions, each against an exact expectation."""
    M, N, K = 9, 11, 13
    A = synth.matrix(M, K, seed=71, stream=0, dist="int")
    B = synth.matrix(K, N, seed=71, stream=1, dist="int")
    C0 = synth.matrix(M, N, seed=71, stream=2, dist="int")
    AB = (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float32)
    nan = np.full((M, N), np.nan, dtype=np.float32)
    # beta == 0: C0 is not read, NaN in C0 does not propagate.
    assert np.array_equal(orc.sgemm(A, B, nan, beta=0.0), AB), "beta=0 read C0"
    # beta == 1 accumulates; beta == 0.5 halves C0 exactly.
    assert np.array_equal(orc.sgemm(A, B, C0, beta=1.0), AB + C0), "beta=1 accumulate"
    assert np.array_equal(orc.sgemm(A, B, C0, beta=0.5), AB + np.float32(0.5) * C0), \
        "beta=0.5 accumulate"
    # alpha == 0: A and B are not read; C = beta*C0.
    An = np.full((M, K), np.nan, dtype=np.float32)
    Bn = np.full((K, N), np.nan, dtype=np.float32)
    assert np.array_equal(orc.sgemm(An, Bn, C0, alpha=0.0, beta=-2.0), -2 * C0), \
        "alpha=0 read A or B"
    # K == 0: the sum is empty; C = beta*C0.
    A0 = np.zeros((M, 0), dtype=np.float32)
    B0 = np.zeros((0, N), dtype=np.float32)
    assert np.array_equal(orc.sgemm(A0, B0, C0, alpha=3.0, beta=0.25),
                          np.float32(0.25) * C0), "K=0"
    # Negative alpha flips the sign exactly.
    assert np.array_equal(orc.sgemm(A, B, alpha=-1.0), -AB), "alpha=-1"
    # A power-of-two alpha scales exactly.
    Af = synth.matrix(M, K, seed=72, stream=0, dist="normal")
    Bf = synth.matrix(K, N, seed=72, stream=1, dist="normal")
    assert np.array_equal(orc.sgemm(Af, Bf, alpha=4.0), 4 * orc.sgemm(Af, Bf)), "alpha=4"


def pin_ld_gaps(orc):
    """Row-strided operands whose gap columns hold NaN: results must equal the
    dense copies' results bit for bit, so no gap element is ever read."""
    M, N, K = 14, 10, 22
    A = synth.matrix(M, K, seed=81, stream=0, dist="normal", ld=K + 5)
    B = synth.matrix(K, N, seed=81, stream=1, dist="normal", ld=N + 3)
    C0 = synth.matrix(M, N, seed=81, stream=2, dist="normal", ld=N + 7)
    got = orc.sgemm(A, B, C0, alpha=0.5, beta=2.0)
    want = orc.sgemm(A.copy(), B.copy(), C0.copy(), alpha=0.5, beta=2.0)
    assert np.isfinite(got).all(), "a NaN gap column was read"
    assert np.array_equal(got, want), "strided and dense results differ"


def pin_row_subset(orc):
    """The row-subset entry returns exactly the selected rows of the full result."""
    M, N, K = 40, 12, 18
    A = synth.matrix(M, K, seed=91, stream=0, dist="normal")
    B = synth.matrix(K, N, seed=91, stream=1, dist="normal")
    C0 = synth.matrix(M, N, seed=91, stream=2, dist="normal")
    full = orc.sgemm(A, B, C0, alpha=1.0, beta=0.5)
    rows = np.array([39, 0, 17, 17, 5])
    assert np.array_equal(orc.sgemm(A, B, C0, alpha=1.0, beta=0.5, rows=rows), full[rows])


def _f32(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def pin_tf32_exact_cases(orc):
    """TF32 rounding (10 stored mantissa bits, nearest, ties away from zero) on
    hand-computed cases: values already in TF32, values just below / at / just
    above a tie, a tie whose even neighbour is the lower one, a carry into the
    next binade, overflow past the largest TF32 value, signed zeros and the
    special values."""
    u = 2.0 ** -23
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0 ** -10, 1.0 + 2.0 ** -10),                 # representable
        (1.0 + 2.0 ** -11, 1.0 + 2.0 ** -10),                 # tie: away from zero
        (1.0 + 2.0 ** -11 - u, 1.0),                          # just below the tie
        (1.0 + 2.0 ** -11 + u, 1.0 + 2.0 ** -10),             # just above the tie
        (-(1.0 + 2.0 ** -11), -(1.0 + 2.0 ** -10)),           # tie, negative: away
        (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),              # tie; the even neighbour is below
        (2.0 - u, 2.0),                                       # carry into the next binade
        (3.0 * 2.0 ** -130, 3.0 * 2.0 ** -130),               # subnormal, representable
        ((2.0 - 2.0 ** -10) * 2.0 ** 127, (2.0 - 2.0 ** -10) * 2.0 ** 127),   # largest TF32
        (float(np.finfo(np.float32).max), np.inf),            # above it: overflow
        (np.inf, np.inf), (-np.inf, -np.inf),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.float32)
    got = orc.round_tf32(x)
    assert np.array_equal(got, want), (x, got, want)
    z = orc.round_tf32(np.array([0.0, -0.0], dtype=np.float32))
    assert z[0] == 0 and not np.signbit(z[0]) and z[1] == 0 and np.signbit(z[1])
    nan = orc.round_tf32(np.array([np.nan, _f32(0x7f800001), _f32(0xff800001)], dtype=np.float32))
    assert np.all(np.isnan(nan))


def pin_tf32_nearest(orc):
    """On random normal floats of every exponent the result is a TF32 value,
    it is one of the two TF32 values around x (x cut toward zero to 10 stored
    bits, and that plus one TF32 step away from zero), it is at least as close
    to x as the other one in exact fp64 arithmetic, and on a tie it is the one
    farther from zero."""
    rng = _rng(97)
    bits = rng.integers(0x00800000, 0x7f000000, size=200000, dtype=np.uint32)
    bits |= rng.integers(0, 2, size=bits.size, dtype=np.uint32) << 31
    bits[:2000] = (bits[:2000] & 0xffffe000) | 0x1000          # exact ties
    x = bits.view(np.float32)
    r = orc.round_tf32(x)
    assert np.all((r.view(np.uint32) & 0x1fff) == 0), "result has more than 10 stored bits"
    cut = (bits & 0xffffe000).view(np.float32).astype(np.float64)      # toward zero
    e = np.floor(np.log2(np.abs(cut)))
    up = cut + np.sign(cut) * np.exp2(e - 10)                          # one TF32 step away
    xd, rd = x.astype(np.float64), r.astype(np.float64)
    assert np.all((rd == cut) | (rd == up)), "not a neighbour of x"
    d_r, d_o = np.abs(xd - rd), np.abs(xd - np.where(rd == cut, up, cut))
    assert np.all(d_r <= d_o), "not the nearest neighbour"
    tie = d_r == d_o
    assert tie[:2000].all() and np.all(np.abs(rd[tie]) > np.abs(xd[tie])), "tie not away from zero"


def pin_bf16_exact_cases(orc):
    """BF16 rounding (7 stored mantissa bits, nearest, ties to even) on
    hand-computed cases, including ties in both directions and the carry."""
    u = 2.0 ** -23
    cases = [
        (1.0, 1.0),
        (1.0 + 2.0 ** -7, 1.0 + 2.0 ** -7),                   # representable
        (1.0 + 2.0 ** -8, 1.0),                               # tie, even neighbour below
        (1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -6),               # tie, even neighbour above
        (1.0 + 2.0 ** -8 + u, 1.0 + 2.0 ** -7),               # just above a tie
        (1.0 + 3 * 2.0 ** -8 - u, 1.0 + 2.0 ** -7),           # just below a tie
        (-(1.0 + 3 * 2.0 ** -8), -(1.0 + 2.0 ** -6)),         # negative tie, to even
        (2.0 - u, 2.0),                                       # carry into the next binade
        ((2.0 - 2.0 ** -7) * 2.0 ** 127, (2.0 - 2.0 ** -7) * 2.0 ** 127),   # largest BF16
        (float(np.finfo(np.float32).max), np.inf),
        (np.inf, np.inf), (-np.inf, -np.inf),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.float32)
    assert np.array_equal(orc.round_bf16(x), want), (x, orc.round_bf16(x), want)
    nan = orc.round_bf16(np.array([np.nan, _f32(0x7f800001)], dtype=np.float32))
    assert np.all(np.isnan(nan))


def pin_bf16_nearest(orc):
    """Random normal floats: the result has 7 stored bits, is one of x's two
    BF16 neighbours, the nearer in exact fp64 distance, and on a tie the one
    whose last kept bit is 0."""
    rng = _rng(98)
    bits = rng.integers(0x00800000, 0x7f000000, size=200000, dtype=np.uint32)
    bits |= rng.integers(0, 2, size=bits.size, dtype=np.uint32) << 31
    bits[:2000] = (bits[:2000] & 0xffff0000) | 0x8000            # exact ties
    x = bits.view(np.float32)
    r = orc.round_bf16(x)
    rb = r.view(np.uint32)
    assert np.all((rb & 0xffff) == 0)
    cut = (bits & 0xffff0000).view(np.float32).astype(np.float64)
    e = np.floor(np.log2(np.abs(cut)))
    up = cut + np.sign(cut) * np.exp2(e - 7)
    xd, rd = x.astype(np.float64), r.astype(np.float64)
    assert np.all((rd == cut) | (rd == up))
    d_r, d_o = np.abs(xd - rd), np.abs(xd - np.where(rd == cut, up, cut))
    assert np.all(d_r <= d_o)
    tie = d_r == d_o
    assert tie[:2000].all() and np.all(((rb[tie] >> 16) & 1) == 0), "tie not to even"


def pin_bias_relu(orc):
    """Fused epilogue on small integers, exact in int64: the bias is per column
    (added to every row), ReLU clamps the sum below zero, and a NaN in C0
    reaches the output through ReLU (it is not clamped to 0)."""
    M, N, K = 23, 17, 30
    A = synth.matrix(M, K, seed=101, stream=0, dist="int")
    B = synth.matrix(K, N, seed=101, stream=1, dist="int")
    C0 = synth.matrix(M, N, seed=101, stream=2, dist="int")
    bias = synth.matrix(1, N, seed=101, stream=3, dist="int")[0] * 8
    exact = (A.astype(np.int64) @ B.astype(np.int64) * 2 - C0.astype(np.int64)
             + bias.astype(np.int64)[None, :])
    got = orc.sgemm(A, B, C0, alpha=2.0, beta=-1.0, bias=bias)
    assert np.array_equal(got, exact.astype(np.float32))
    got = orc.sgemm(A, B, C0, alpha=2.0, beta=-1.0, bias=bias, act="relu")
    assert np.array_equal(got, np.maximum(exact, 0).astype(np.float32))
    assert (exact < 0).any() and (exact > 0).any()
    C1 = C0.copy()
    C1[3, 4] = np.nan
    got = orc.sgemm(A, B, C1, alpha=1.0, beta=1.0, act="relu")
    assert np.isnan(got[3, 4]) and np.isfinite(np.delete(got.reshape(-1), 3 * N + 4)).all()
    # alpha = 0: act(beta*C0 + bias), A and B not read
    got = orc.sgemm(np.full((M, K), np.nan, np.float32), np.full((K, N), np.nan, np.float32), C0,
                    alpha=0.0, beta=1.0, bias=bias, act="relu")
    assert np.array_equal(got, np.maximum(C0.astype(np.int64) + bias[None, :], 0).astype(np.float32))


def _act_inputs(orc):
    """x values from -12 to 12 as the rows of A @ I (exact)."""
    x = np.linspace(-12.0, 12.0, 481, dtype=np.float32).reshape(1, -1)
    return x, np.eye(1, dtype=np.float32)


def pin_gelu_silu(orc):
    """GELU (tanh form) and SiLU on x in [-12, 12], checked against other
    formulas, not their own: both satisfy f(x) - f(-x) = x (their "gates" g
    obey g(x) + g(-x) = 1); GELU's tanh form stays within 1e-3 of the exact
    erf form x*Phi(x); SiLU equals x*(1 + tanh(x/2))/2; and both tend to x for
    large x and to 0 for large negative x."""
    import math
    x, eye = _act_inputs(orc)
    xs = x.reshape(-1).astype(np.float64)
    for act in ("gelu", "silu"):
        f = orc.sgemm(eye, x, act=act).reshape(-1).astype(np.float64)       # f(x)
        g = orc.sgemm(eye, -x, act=act).reshape(-1).astype(np.float64)      # f(-x)
        tol = 4 * 2.0 ** -24 * np.maximum(np.abs(f), np.abs(g)) + 1e-30
        assert np.all(np.abs((f - g) - xs) <= tol + 2.0 ** -24 * np.abs(xs)), act
        assert abs(f[-1] - 12.0) < 1e-4 and abs(f[0]) < 1e-4, act   # 12*sigmoid(-12) = 7.4e-5
    gelu = orc.sgemm(eye, x, act="gelu").reshape(-1).astype(np.float64)
    exact = np.array([v * 0.5 * (1.0 + math.erf(v / math.sqrt(2.0))) for v in xs])
    assert np.max(np.abs(gelu - exact)) < 1e-3
    assert np.max(np.abs(gelu - exact)) > 1e-5     # the tanh form, not the erf form
    silu = orc.sgemm(eye, x, act="silu").reshape(-1).astype(np.float64)
    other = xs * (1.0 + np.tanh(xs / 2.0)) / 2.0
    assert np.all(np.abs(silu - other) <= 2.0 ** -22 * np.abs(other) + 1e-30)


ALL_PINS = [pin_small_int_exact, pin_exact_rational, pin_identity, pin_permutation,
            pin_rank1, pin_transpose, pin_freivalds, pin_alpha_beta, pin_ld_gaps,
            pin_row_subset, pin_tf32_exact_cases, pin_tf32_nearest, pin_bf16_exact_cases,
            pin_bf16_nearest, pin_bias_relu, pin_gelu_silu]
