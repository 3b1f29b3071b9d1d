"""Pins of the oracle's deterministic index_add (Megatron-LM PR #7441, Source 3).

Independent checks: the sort against numpy's stable argsort and the segment
offsets against bincount, seg_tile = 1 against numpy's in-order add.at
(bitwise, zero-initialised out), exact integer sums on ternary inputs, fp64
sums within the error bound, padding and out-of-range routing to the dummy
row, and untouched empty rows.
"""
import math

import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal, gamma, rel_l2


def _run(ia: gi.IndexAddInput, seg_tile=128):
    out = gi.f32(ia.out).copy()
    src = gi.f32(ia.src)
    N, D = src.shape
    bad, perm, seg = oracle.det_index_add(out, ia.R, D, D, src, D, ia.idx.numpy(), N, seg_tile=seg_tile)
    return out, bad, perm, seg


def _keys(idx, R):
    k = idx.astype(np.int64).copy()
    k[(k < 0) | (k >= R)] = R
    return k


@pytest.mark.parametrize("N,D,R", [(20000, 16, 500), (3000, 8, 3), (5000, 4, 0), (1, 4, 10)])
def test_sort_matches_stable_argsort(N, D, R):
    ia = gi.index_add_input(N, D, R, seed=31)
    _, bad, perm, seg = _run(ia)
    k = _keys(ia.idx.numpy(), R)
    assert bad == 0
    np.testing.assert_array_equal(perm, np.argsort(k, kind="stable"))
    cnt = np.bincount(k, minlength=R + 1)
    np.testing.assert_array_equal(seg, np.concatenate([[0], np.cumsum(cnt)]))


def test_seg_tile_one_is_in_order_add_at():
    ia = gi.index_add_input(30000, 8, 700, seed=32)
    got, *_ = _run(ia, seg_tile=1)
    want = gi.f32(ia.out).copy()
    k = _keys(ia.idx.numpy(), ia.R)
    np.add.at(want, k, gi.f32(ia.src))
    assert_bits_equal(got, want, "seg_tile=1 vs np.add.at")


@pytest.mark.parametrize("seg_tile", [1, 4, 128])
def test_ternary_exact_with_integer_init(seg_tile):
    ia = gi.index_add_input(40000, 8, 300, seed=33, dist="ternary", out_init="random")
    out0 = torch.round(ia.out * 3).numpy().astype(np.float32)
    ia = gi.IndexAddInput(ia.src, ia.idx, torch.from_numpy(out0), ia.R)
    got, *_ = _run(ia, seg_tile=seg_tile)
    want = out0.astype(np.int64)
    np.add.at(want, _keys(ia.idx.numpy(), ia.R), gi.f32(ia.src).astype(np.int64))
    assert_bits_equal(got, want.astype(np.float32), "ternary index_add")


def test_fp64_bound_and_dummy_row():
    ia = gi.index_add_input(50000, 16, 64, seed=34)
    got, *_ = _run(ia)
    k = _keys(ia.idx.numpy(), ia.R)
    src = gi.f32(ia.src).astype(np.float64)
    exact = np.zeros((ia.R + 1, 16))
    np.add.at(exact, k, src)
    absum = np.zeros((ia.R + 1, 16))
    np.add.at(absum, k, np.abs(src))
    cnt = np.bincount(k, minlength=ia.R + 1)
    kbound = np.array([int(math.log2(128)) + -(-c // 128) + 1 for c in cnt])[:, None]
    bound = np.vectorize(gamma)(kbound) * absum
    assert np.all(np.abs(got - exact) <= bound)
    assert rel_l2(got, exact) <= 1e-5
    assert cnt[ia.R] == int(0.1 * 50000)  # padding went to the dummy row


def test_bad_indices_are_counted_and_routed_to_dummy():
    ia = gi.index_add_input(1000, 4, 50, seed=35, pad_frac=0.0)
    idx = ia.idx.clone()
    idx[[3, 10, 500]] = torch.tensor([50, -2, 1 << 30], dtype=torch.int32)
    idx[7] = -1
    ib = gi.IndexAddInput(ia.src, idx, ia.out, ia.R)
    got, bad, perm, seg = _run(ib)
    assert bad == 3
    assert seg[ia.R + 1] - seg[ia.R] == 4
    assert sorted(perm[seg[ia.R]:seg[ia.R + 1]].tolist()) == [3, 7, 10, 500]


def test_empty_rows_untouched_and_signed_zero():
    ia = gi.index_add_input(200, 4, 1000, seed=36, out_init="random")
    out0 = gi.f32(ia.out).copy()
    out0[5] = -0.0
    ia = gi.IndexAddInput(ia.src, ia.idx, torch.from_numpy(out0), ia.R)
    got, *_ = _run(ia)
    used = np.zeros(ia.R + 1, bool)
    used[_keys(ia.idx.numpy(), ia.R)] = True
    assert_bits_equal(got[~used], out0[~used], "untouched rows")


def test_empty_input():
    ia = gi.index_add_input(0, 4, 10, seed=37, out_init="random")
    out0 = gi.f32(ia.out).copy()
    got, bad, _, seg = _run(ia)
    assert bad == 0 and np.all(seg == 0)
    assert_bits_equal(got, out0, "N=0")
