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


def test_packed_product_feeding_scalar_adds_keeps_both_roundings():
    # the dsReLU leaves' form: c + RN(a * b) with the product packed and the add
    # scalar equals two separately rounded float32 operations (no fusion)
    n = 1 << 22
    rng = np.random.default_rng(11)
    a, b, c = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    A, B, C = (torch.from_numpy(x).cuda() for x in (a, b, c))
    out = torch.empty_like(A)
    assert dgr.lib().dgr_diag_packed_chain(A.data_ptr(), B.data_ptr(), C.data_ptr(), n // 2, out.data_ptr(), None) == 0
    want = c + (a * b)  # numpy float32: the product rounded, then the sum rounded
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    fused = (a.astype(np.float64) * b + c).astype(np.float32)  # one rounding, as a fused multiply-add would give
    assert (fused.view(np.uint32) != want.view(np.uint32)).sum() > n // 20  # the case can tell them apart
