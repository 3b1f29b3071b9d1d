"""Pins of the oracle's tree and fold: hand-derived cases and identities.

These run on the CPU only and pin the canonical order itself: the pairing of
the pairwise tree, the rule for absent leaves in a ragged tile, the ascending
fold and the single-rounding accumulate.
"""
import numpy as np
import pytest

import oracle
from util import assert_bits_equal, load_hand_cases

CASES = load_hand_cases()


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_hand_cases(case):
    kind, width, vals, expected, _passage = case
    if kind == "pairwise":
        got = oracle.pairwise(vals, width)
    elif kind == "fold":
        got = oracle.fold(vals)
    elif kind == "accum":
        # out + F through the column-sum entry: one tile holding F, accumulate on
        out = np.array([vals[0]], np.float32)
        x = np.array([vals[1]], np.float32)
        oracle.ordered_colsum(x, 1, 1, 1, 1, 1, out, accumulate=True, tile_rows=1)
        got = out[0]
    else:  # pragma: no cover
        raise AssertionError(kind)
    assert_bits_equal(got, expected, f"{kind} {vals.tolist()}")


def test_hand_cases_cover_every_kind():
    assert {c[0] for c in CASES} == {"pairwise", "fold", "accum"}
    assert len(CASES) >= 7


def test_single_leaf_is_itself():
    rng = np.random.default_rng(0)
    for w in (1, 2, 8, 128):
        v = rng.standard_normal(1).astype(np.float32)
        assert_bits_equal(oracle.pairwise(v, w), v[0])


def test_width_one_tiles_are_a_sequential_fold():
    # With one leaf per tile the canonical order is the plain sequential sum,
    # which numpy's add.accumulate computes step by step in float32.
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(1000) * np.exp(rng.uniform(-8, 8, 1000))).astype(np.float32)
    want = np.add.accumulate(v, dtype=np.float32)[-1]
    out = np.zeros(1, np.float32)
    oracle.ordered_colsum(v, 1, v.size, 1, v.size, 1, out, tile_rows=1)
    assert_bits_equal(out[0], want, "tile_rows=1")
    assert_bits_equal(oracle.fold(v), want, "fold")


def test_ragged_tile_equals_padding_with_negative_zero():
    # Absent leaves pass the other child through, which is what -0.0 padding
    # does under round-to-nearest (x + -0.0 == x for every x, including -0.0).
    rng = np.random.default_rng(2)
    for count in (1, 3, 5, 7, 100, 127):
        v = rng.standard_normal(count).astype(np.float32)
        padded = np.concatenate([v, np.full(128 - count, -0.0, np.float32)])
        assert_bits_equal(oracle.pairwise(v, 128), oracle.pairwise(padded, 128), f"count {count}")


def test_pairwise_exact_on_integers_any_width():
    # integer leaves with small sums: every order is exact
    rng = np.random.default_rng(3)
    for w in (2, 16, 128, 1024):
        v = rng.integers(-1000, 1000, w).astype(np.float32)
        assert oracle.pairwise(v, w) == np.float32(v.astype(np.int64).sum())


def test_pairwise_is_not_sequential_on_adversarial_data():
    # the oracle must not silently be a running sum: 2^24 followed by ones
    v = np.array([2.0 ** 24] + [1.0] * 127, np.float32)
    seq = np.add.accumulate(v, dtype=np.float32)[-1]
    assert seq == np.float32(2.0 ** 24)
    assert oracle.pairwise(v, 128) == np.float32(2.0 ** 24 + 126)
