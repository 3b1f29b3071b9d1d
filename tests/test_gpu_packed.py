"""The packed binary32 add and multiply (add.rn.f32x2, mul.rn.f32x2) that the
kernels use in place of pairs of scalar round-to-nearest operations, pinned
bit for bit against numpy's float32 arithmetic (IEEE 754 round to nearest
even, subnormals kept) on operands drawn so that many inputs and results are
subnormal, exact ties or cancellations, or overflow. NaN results need only be
NaN."""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr

pytestmark = pytest.mark.gpu


def _operands(n: int, seed: int):
    rng = np.random.default_rng(seed)
    u = lambda k: rng.integers(0, 1 << 32, k, dtype=np.uint64).astype(np.uint32)
    a, b = u(n), u(n)
    q = n // 4
    a[:q] &= 0x807FFFFF                                   # subnormal with subnormal
    b[:q] &= 0x807FFFFF
    e = rng.integers(1, 254, q).astype(np.uint32) << 23   # equal exponents: ties and cancellations
    a[q:2 * q] = (a[q:2 * q] & 0x807FFFFF) | e
    b[q:2 * q] = (b[q:2 * q] & 0x807FFFFF) | e
    e1 = rng.integers(0, 255, q).astype(np.uint32) << 23  # products over the whole exponent range
    e2 = rng.integers(0, 255, q).astype(np.uint32) << 23
    a[2 * q:3 * q] = (a[2 * q:3 * q] & 0x807FFFFF) | e1
    b[2 * q:3 * q] = (b[2 * q:3 * q] & 0x807FFFFF) | e2
    return a.view(np.float32), b.view(np.float32)        # the last quarter: any bits


def test_packed_add_and_mul_match_ieee_float32():
    n = 1 << 22
    a, b = _operands(n, 7)
    A, B = torch.from_numpy(a.copy()).cuda(), torch.from_numpy(b.copy()).cuda()
    S, M = torch.empty_like(A), torch.empty_like(A)
    rc = dgr.lib().dgr_diag_packed_ops(A.data_ptr(), B.data_ptr(), n // 2, S.data_ptr(), M.data_ptr(), None)
    assert rc == 0
    s, m = S.cpu().numpy(), M.cpu().numpy()
    with np.errstate(all="ignore"):
        ws, wm = a + b, a * b
    for got, want, what in ((s, ws, "add"), (m, wm, "mul")):
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan), what
        diff = (got.view(np.uint32) != want.view(np.uint32)) & ~nan
        assert not diff.any(), f"{what}: {int(diff.sum())} of {n} differ"
        sub = ((want.view(np.uint32) & 0x7F800000) == 0) & (want != 0)
        assert sub.sum() > n // 50, what  # the draw did reach subnormal results (3 % of products, 19 % of sums)
