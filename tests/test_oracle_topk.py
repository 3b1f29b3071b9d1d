"""Pins of the oracle's canonical compact top-K (Megatron-LM PR #7441, Source 1).

Independent checks: the permutation equals numpy's stable argsort with
padding keyed last; every output row is bitwise the same whatever order its
slots come in (the point of the fix: nothing may depend on the slot order);
the probabilities match an fp64 softmax of the valid logits to a few ulps and
sum to one; special cases: one valid slot gives exactly 1, an all-padding row
gives +0.0 everywhere, padding slots get +0.0.
"""
import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal


def _np_perm(ids: np.ndarray) -> np.ndarray:
    key = np.where(ids < 0, np.int64(2) ** 40, ids.astype(np.int64))
    return np.argsort(key, axis=1, kind="stable")


@pytest.mark.parametrize("R,K", [(300, 128), (200, 64), (100, 256), (50, 7)])
def test_permutation_is_the_stable_sort(R, K):
    t = gi.topk_input(R, K, seed=41 + K, n_keys=4096)
    ids, lg = t.ids.numpy(), t.logits.numpy()
    oi, ol, _ = oracle.topk_canonicalize(ids, lg)
    perm = _np_perm(ids)
    assert np.array_equal(oi, np.take_along_axis(ids, perm, 1))
    assert_bits_equal(ol, np.take_along_axis(lg, perm, 1), "permuted logits")


@pytest.mark.parametrize("K", [128, 256, 33])
def test_outputs_do_not_depend_on_the_slot_order(K):
    t = gi.topk_input(400, K, seed=42, n_keys=8192)
    ids, lg = t.ids.numpy(), t.logits.numpy()
    ref = oracle.topk_canonicalize(ids, lg)
    rng = np.random.default_rng(5)
    for _ in range(3):
        order = np.argsort(rng.random(ids.shape), axis=1)
        # a permutation of the valid slots only: padding slots keep their
        # relative order (their logits are carried along, so moving them
        # among themselves would permute what they carry)
        got = oracle.topk_canonicalize(np.take_along_axis(ids, order, 1), np.take_along_axis(lg, order, 1))
        valid_rows = ~(ids < 0).any(axis=1)
        assert np.array_equal(got[0], ref[0])
        for a, b in zip(got[1:], ref[1:]):
            assert_bits_equal(a[valid_rows], b[valid_rows], "slot order")
        # probabilities never depend on the padding slots at all
        assert_bits_equal(got[2], ref[2], "probs")


def test_probabilities_match_fp64_softmax():
    t = gi.topk_input(1000, 128, seed=43, n_keys=65536)
    ids, lg = t.ids.numpy(), t.logits.numpy()
    oi, ol, pr = oracle.topk_canonicalize(ids, lg)
    valid = oi >= 0
    x = np.where(valid, ol.astype(np.float64), -np.inf)
    m = x.max(axis=1, keepdims=True)
    with np.errstate(invalid="ignore"):
        e = np.exp(x - m)
        p64 = e / e.sum(axis=1, keepdims=True)
    p64 = np.where(valid, p64, 0.0)
    rows = valid.any(axis=1)
    rel = np.abs(pr[rows] - p64[rows]) / np.maximum(p64[rows], 1e-30)
    # d = RN(l - m) is off by up to 2^-24 |d|, which exp turns into the same
    # relative error; then the exponential's own error (at most 0.77 ulp,
    # 1.54 * 2^-24 relative, in e and in every term of Z), the tree over <= 128
    # positive terms (7 levels) and the division: 2^-24 (|d_k| + max |d| + 12)
    d = np.abs(np.where(valid, ol.astype(np.float64) - m, 0.0))
    bound = 2.0 ** -24 * (d + d.max(axis=1, keepdims=True) + 12)
    assert np.all(rel[valid[rows]] <= bound[rows][valid[rows]])
    assert np.all(np.abs(pr[rows].astype(np.float64).sum(axis=1) - 1.0) <= 128 * 2.0 ** -23)
    assert not np.any(pr[~valid]) and not np.any(np.signbit(pr[~valid]))


def test_special_rows():
    ids = np.array([[-1, -1, -1, -1], [-1, 7, -1, -1], [3, 1, 2, 0]], np.int32)
    lg = np.array([[1, 2, 3, 4], [9, -5.5, 1, 1], [0, 0, 0, 0]], np.float32)
    oi, ol, pr = oracle.topk_canonicalize(ids, lg)
    assert not np.any(pr[0]) and not np.any(np.signbit(pr[0]))      # all padding: 0, not NaN
    assert np.array_equal(oi[0], ids[0]) and np.array_equal(ol[0], lg[0])  # padding keeps its order
    assert pr[1, 0] == 1.0 and not np.any(pr[1, 1:])                 # one valid slot
    assert np.array_equal(oi[1], [7, -1, -1, -1]) and np.array_equal(ol[1], [-5.5, 9, 1, 1])
    assert np.array_equal(oi[2], [0, 1, 2, 3])
    assert np.all(pr[2] == np.float32(0.25))                         # equal logits: exactly 1/4


def _ulps(got: np.ndarray, x: np.ndarray) -> np.ndarray:
    exact = np.exp(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(exact, 1e-300)))
    ulp = np.maximum(2.0 ** (e - 23), 2.0 ** -149)  # binary32 ulp of the exact value (subnormal floor)
    return np.abs(got.astype(np.float64) - exact) / ulp


def test_exponential_table_is_two_to_the_j_over_32():
    # Tang's table: S_lead[j] is 2^(j/32) rounded to 18 significant bits and
    # S_trail[j] the rest rounded to binary32, here recomputed in exact decimal
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    lead, trail = oracle.exp_tang_constants()
    for j in range(32):
        s = Decimal(2) ** (Decimal(j) / 32)
        sl = (s * 2 ** 17).to_integral_value() / Decimal(2 ** 17)
        assert Decimal(float(lead[j])) == sl, j
        rest = s - sl
        t = Decimal(float(trail[j]))
        # the binary32 nearest the rest: within half a binary32 ulp of it
        half_ulp = Decimal(2) ** (int(np.floor(np.log2(abs(float(rest))))) - 24) if rest != 0 else Decimal(0)
        assert abs(t - rest) <= half_ulp, j


def test_exponential_accuracy_and_special_values():
    # within 0.77 ulp of exp (the exhaustive measurement over [-104, 0]) on a
    # large seeded sample, bit patterns spaced evenly over the whole range
    # and uniform values, and exact where exp is exact
    rng = np.random.default_rng(71)
    lo, hi = 0x80000000, int(np.float32(-104.0).view(np.uint32))
    even = np.linspace(lo, hi, 1 << 21, dtype=np.float64).astype(np.uint64).astype(np.uint32).view(np.float32)
    uni = rng.uniform(-104.0, 0.0, 1 << 21).astype(np.float32)
    small = -rng.uniform(0.0, 0.02, 1 << 18).astype(np.float32)  # around the table points, |r| small
    for x in (even, uni, small):
        err = _ulps(oracle.exp_tang(x), x)
        assert err.max() <= 0.77, (float(err.max()), float(x[np.argmax(err)]))
    got = oracle.exp_tang(np.array([0.0, -0.0, -104.5, -1e30, np.nan], np.float32))
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 0.0 and got[3] == 0.0 and np.isnan(got[4])
