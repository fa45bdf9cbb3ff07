"""Helpers for the GPU parity tests: padded device copies with canaries, the
normwise error of the acceptance gate, and one checked library call."""

from __future__ import annotations

import numpy as np

import oracle
import synth

CANARY_BITS = np.uint32(0x7FC0DEAD)   # a quiet NaN with a recognisable payload
GATE = 1e-6


def normwise_err(C, Cref, A, B, K, alpha=1.0, beta=0.0, C0=None, bias=None):
    """The acceptance gate as a number: <= GATE passes.

    With beta = 0 and no bias this is exactly max|C - C_ref| / (|alpha|*K*
    max|A|*max|B|), the gate on the product.  With beta != 0 or a bias, each
    element may in addition differ by the FP32 rounding of the terms the
    product does not bound, element by element: up to two half-ulp roundings
    (the beta*C + product fma and the bias add) of |beta*C0[i,j]| + |bias[j]|
    + |C_ref[i,j]|, i.e. 2^-22 times that sum.  So element (i,j) passes when

        |C - C_ref| <= GATE*|alpha|*K*max|A|*max|B|
                       + 2^-22 * (|beta*C0[i,j]| + |bias[j]| + |C_ref[i,j]|)

    and the value returned is GATE * max over (i,j) of |C - C_ref| / that
    bound.  The fused activations (ReLU, GELU, SiLU) have slopes below 1.13
    and their own FP32 error is a few ulps of their argument, which the
    product term covers.
    """
    C = np.asarray(C)
    if C.size == 0:
        return 0.0
    amax = float(np.abs(A).max()) if A.size else 0.0
    bmax = float(np.abs(B).max()) if B.size else 0.0
    prod = GATE * abs(alpha) * K * amax * bmax
    extra_terms = (beta != 0.0 and C0 is not None) or bias is not None
    vb = None if bias is None else np.abs(np.asarray(bias, dtype=np.float64)).reshape(1, -1)
    worst = 0.0
    step = max(1, (1 << 22) // max(C.shape[1], 1))       # rows per block (memory bound)
    for r0 in range(0, C.shape[0], step):
        c = C[r0:r0 + step].astype(np.float64)
        cr = Cref[r0:r0 + step].astype(np.float64)
        diff = np.abs(c - cr)
        if np.isnan(diff).any():
            return float("inf")
        bound = np.full(diff.shape, prod)
        if extra_terms:
            t = np.abs(cr)
            if beta != 0.0 and C0 is not None:
                t += abs(beta) * np.abs(C0[r0:r0 + step].astype(np.float64))
            if vb is not None:
                t += vb
            bound += 2.0 ** -22 * t
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(bound > 0, diff / bound, np.where(diff == 0, 0.0, np.inf))
        worst = max(worst, float(ratio.max()))
    return GATE * worst


def product_err(C, Cref, A, B, K, alpha=1.0):
    """max|C - C_ref| / (|alpha|*K*max|A|*max|B|): the gate's metric on the
    product alone (no allowance for beta*C0 or a bias)."""
    if np.asarray(C).size == 0:
        return 0.0
    scale = abs(alpha) * K * float(np.abs(A).max()) * float(np.abs(B).max())
    worst = 0.0
    step = max(1, (1 << 22) // max(C.shape[1], 1))
    for r0 in range(0, C.shape[0], step):
        d = np.abs(C[r0:r0 + step].astype(np.float64) - Cref[r0:r0 + step].astype(np.float64))
        if np.isnan(d).any():
            return float("inf")
        worst = max(worst, float(d.max()))
    return worst / scale if scale > 0 else (0.0 if worst == 0 else float("inf"))


class Padded:
    """A rows x cols matrix in a device buffer with row stride `ld`, starting
    `offset` floats into the buffer, with `guard` canary floats before and
    after and canaries in every gap column."""

    def __init__(self, X: np.ndarray, ld: int | None = None, offset: int = 0, guard: int = 64,
                 device="cuda"):
        import torch
        rows, cols = X.shape
        self.rows, self.cols = rows, cols
        self.ld = max(cols, 1) if ld is None else ld
        self.start = guard + offset
        n = self.start + rows * self.ld + guard
        host = np.full(n, CANARY_BITS, dtype=np.uint32).view(np.float32)
        if rows and cols:
            host[self.start:self.start + rows * self.ld].reshape(rows, self.ld)[:, :cols] = X
        self.template = host.copy()
        self.buf = torch.from_numpy(host).to(device)
        if rows and cols:
            self.view = torch.as_strided(self.buf, (rows, cols), (self.ld, 1), self.start)
        else:
            self.view = torch.empty((rows, cols), dtype=torch.float32, device=device)

    def host(self) -> np.ndarray:
        return self.buf.cpu().numpy()

    def matrix(self, host=None) -> np.ndarray:
        h = self.host() if host is None else host
        if not (self.rows and self.cols):
            return np.zeros((self.rows, self.cols), dtype=np.float32)
        return h[self.start:self.start + self.rows * self.ld].reshape(self.rows, self.ld)[:, :self.cols].copy()

    def outside_intact(self, host=None) -> bool:
        """Every float outside the matrix's own elements still holds its template bits."""
        h = (self.host() if host is None else host).view(np.uint32)
        t = self.template.view(np.uint32)
        if not (self.rows and self.cols):
            return bool(np.array_equal(h, t))
        s, e = self.start, self.start + self.rows * self.ld
        if not (np.array_equal(h[:s], t[:s]) and np.array_equal(h[e:], t[e:])):
            return False
        if self.ld > self.cols:       # the gap columns between rows
            gap = lambda x: x[s:e].reshape(self.rows, self.ld)[:, self.cols:]
            return bool(np.array_equal(gap(h), gap(t)))
        return True

    def unchanged(self) -> bool:
        return bool(np.array_equal(self.host().view(np.uint32), self.template.view(np.uint32)))


def make_inputs(M, N, K, dist="uniform", seed=0, beta=0.0, sigma_b=None):
    sb = 1.0 if sigma_b is None else sigma_b
    A = synth.matrix(M, K, seed=seed, stream=0, dist=dist)
    B = synth.matrix(K, N, seed=seed, stream=1, dist=dist, sigma=sb)
    if beta != 0.0:
        C0 = synth.matrix(M, N, seed=seed, stream=2, dist=dist)
    else:
        C0 = np.full((M, N), np.nan, dtype=np.float32)   # beta == 0 must not read C
    return A, B, C0


def run_checked(sg, A, B, C0, alpha, beta, *, kernel=None, lds=(None, None, None),
                offsets=(0, 0, 0), tensor_cores=False, exact=False, rows=None, bias=None,
                act="none", ref=None, return_c=False):
    """One library call on padded device copies; checks the status, the kernel
    the library chose, canaries around all three operands, and parity with the
    oracle (bit-exact if `exact`, else the normwise gate).  Returns the error
    and the chosen kernel (and the result C if `return_c`).

    `ref` is the oracle's result for these operands (rows `rows` if given),
    when the caller already has it; otherwise it is computed here."""
    M, K = A.shape
    N = B.shape[1]
    if kernel is not None and lds == (None, None, None):
        # give the TMA kernel leading dimensions it can take (multiples of 4);
        # the gap columns hold canaries
        r4 = lambda x: max(4, (x + 3) // 4 * 4)
        lds = (r4(K), r4(N), N + (M % 3))
    pa = Padded(A, lds[0], offsets[0])
    pb = Padded(B, lds[1], offsets[1])
    pc = Padded(C0, lds[2], offsets[2])
    prev = sg.force_kernel(kernel) if kernel is not None else None
    try:
        chosen = sg.select_kernel(M, N, K, alpha, pa.view.data_ptr() or 0, pa.ld,
                                  pb.view.data_ptr() or 0, pb.ld, beta,
                                  pc.view.data_ptr() or 0, pc.ld, tensor_cores)
        import torch
        dbias = torch.from_numpy(bias).cuda() if bias is not None else None
        sg.sgemm(pa.view, pb.view, pc.view, alpha, beta, tensor_cores=tensor_cores, bias=dbias,
                 activation=act)
        st = sg.status()
    finally:
        if prev is not None:
            sg.force_kernel(sg.KERNEL_AUTO)
    assert st == sg.OK, f"kernel status {st}: {sg.status_string(st)}"
    h = pc.host()
    C = pc.matrix(h)
    assert pc.outside_intact(h), "a write landed outside C's elements (gap or guard)"
    assert pa.unchanged() and pb.unchanged(), "A or B was modified"
    use_ab = alpha != 0.0 and K > 0
    # the reduced-precision path is defined on TF32-rounded operands
    inputs = {sg.MODE_TF32: "tf32", sg.MODE_BF16: "bf16"}.get(sg._mode(tensor_cores), "fp32")
    if ref is None:
        Cref = oracle.sgemm(A, B, C0 if beta != 0.0 else None, alpha=alpha, beta=beta, rows=rows,
                            inputs=inputs, bias=bias, act=act)
    else:
        Cref = ref
    got = C if rows is None else C[rows]
    # without the product, beta*C rounds once in both, so the result is exact;
    # not with a bias (beta*C + bias rounds twice in FP32, once in the oracle)
    # or after GELU / SiLU (FP32 tanhf / expf against fp64)
    if exact or (not use_ab and bias is None and act in ("none", "relu")):
        assert np.array_equal(got.view(np.uint32), Cref.view(np.uint32)) or np.array_equal(got, Cref), \
            f"not bit-exact: max |diff| = {np.nanmax(np.abs(got - Cref)) if got.size else 0}"
        err = 0.0
    else:
        err = normwise_err(got, Cref, A, B, K, alpha, beta, C0, bias)
        assert err <= GATE, f"normwise error {err:.3e} above {GATE}"
    if return_c:
        return err, chosen, C
    return err, chosen
