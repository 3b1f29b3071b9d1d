"""Pins of the oracle's ordered dprob (cuDNN-frontend PR #521, "deterministic dprob").

Independent checks: exact integer sums on ternary inputs, the fp64 row dot
within a relative L2 of 1e-5 and the elementwise error bound, the
one-tile and one-column special cases, leading-dimension handling with NaN
poison, and the accumulate convention the page fixes (the slot reduction adds
into dprob like the atomic path it replaces).
"""
import math

import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal, bf16_bits_to_f64, gamma, rel_l2


def _run(di: gi.DprobInput, out=None, **kw):
    ld = di.dY.shape[1]
    out = np.zeros(di.M, np.float32) if out is None else out
    fl = gi.bits if di.dY.dtype == torch.bfloat16 else gi.f32
    slots = oracle.ordered_rowdot_dprob(fl(di.dY).reshape(-1), fl(di.Y).reshape(-1), di.M, di.N, ld, ld,
                                        out, **kw)
    return out, slots


@pytest.mark.parametrize("M,N,ld", [(64, 4096, None), (33, 1000, 1024), (5, 129, None)])
def test_ternary_exact(M, N, ld):
    di = gi.dprob_input(M, N, seed=21, dist="ternary", ld=ld)
    a = di.dY[:, :N].to(torch.int64).numpy()
    b = di.Y[:, :N].to(torch.int64).numpy()
    got, _ = _run(di)
    assert_bits_equal(got, (a * b).sum(axis=1).astype(np.float32), "ternary dprob")


@pytest.mark.parametrize("W", [16, 128, 512])
def test_fp64_bound(W):
    di = gi.dprob_input(128, 4096, seed=22)
    a = di.dY.to(torch.float64).numpy()
    b = di.Y.to(torch.float64).numpy()
    exact = (a * b).sum(axis=1)
    got, _ = _run(di, tile_n=W)
    k = 1 + int(math.log2(W)) + -(-4096 // W)  # the product rounding, the tree, the fold
    bound = gamma(k) * np.abs(a * b).sum(axis=1)
    assert np.all(np.abs(got.astype(np.float64) - exact) <= bound)
    assert rel_l2(got, exact) <= 1e-5


def test_single_column_is_the_rounded_product():
    # N = 1: dprob = RN(dY * Y), the one multiply rounded on its own
    di = gi.dprob_input(1000, 1, seed=23, dtype=torch.float32)
    got, _ = _run(di)
    want = (gi.f32(di.dY)[:, 0] * gi.f32(di.Y)[:, 0]).astype(np.float32)
    assert_bits_equal(got, want, "N=1")


def test_slots_hold_tile_partials_and_fold_ascending():
    di = gi.dprob_input(4, 1000, seed=24)
    got, slots = _run(di, return_slots=True)
    assert slots.shape == (4, 8)
    p = (bf16_bits_to_f64(gi.bits(di.dY)) * bf16_bits_to_f64(gi.bits(di.Y))).astype(np.float32)
    p = p.reshape(4, 1000)
    for m in range(4):
        for j in (0, 7):
            assert_bits_equal(slots[m, j], oracle.pairwise(p[m, j * 128:(j + 1) * 128], 128))
        assert_bits_equal(got[m], oracle.fold(slots[m]))


def test_leading_dimension_skips_poison():
    di = gi.dprob_input(16, 300, seed=25, ld=512)
    got, _ = _run(di)
    assert np.all(np.isfinite(got))
    dense = gi.DprobInput(di.dY[:, :300].contiguous(), di.Y[:, :300].contiguous(), 16, 300)
    assert_bits_equal(got, _run(dense)[0], "ld vs dense")


def test_accumulate_and_empty():
    di = gi.dprob_input(32, 777, seed=26)
    fresh, _ = _run(di)
    d0 = np.random.default_rng(5).standard_normal(32).astype(np.float32)
    acc, _ = _run(di, out=d0.copy(), accumulate=True)
    assert_bits_equal(acc, (d0 + fresh).astype(np.float32), "accumulate")
    empty = gi.DprobInput(di.dY, di.Y, 32, 0)
    o, _ = _run(empty, out=np.full(32, 3.0, np.float32))
    assert_bits_equal(o, np.zeros(32, np.float32), "N=0 overwrite")
    o, _ = _run(empty, out=np.full(32, 3.0, np.float32), accumulate=True)
    assert_bits_equal(o, np.full(32, 3.0, np.float32), "N=0 accumulate")
