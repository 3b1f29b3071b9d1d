"""Pins of the oracle's grouped dbias (cuDNN-frontend PR #521, commit "Cover dbias").

dbias[e] is an ordered column sum over expert e's rows, its tiles counted
from the expert's first row. Independent checks: exact integer sums per expert
(ternary inputs make every partial an integer below 2^24, so every order gives
the exact int64 sum), agreement with the separately pinned column sum run on
each expert's row slice, the fp64 sum within the pairwise error bound, a
hand-worked case where tiles counted from the expert's start and tiles counted
from row 0 give different bits, the one-rounding accumulate, empty experts,
and NaN poison past H in strided rows.
"""
import math

import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal, gamma, rel_l2


def _flat(d: gi.DbiasInput) -> np.ndarray:
    return gi.bits(d.dY).reshape(-1) if d.dY.dtype == torch.bfloat16 else gi.f32(d.dY).reshape(-1)


def _run(d: gi.DbiasInput, out0=None, **kw) -> np.ndarray:
    out = np.zeros(d.E * d.H, np.float32) if out0 is None else out0.reshape(-1).copy()
    oracle.grouped_dbias(_flat(d), d.T, d.H, d.ld, d.offs.numpy(), out, **kw)
    return out.reshape(d.E, d.H)


def _rows64(d: gi.DbiasInput) -> np.ndarray:
    return d.dY[:, :d.H].to(torch.float64).numpy()


@pytest.mark.parametrize("T,H,E,ld", [(5000, 16, 4, None), (3000, 24, 7, 40), (65536, 2048, 8, None)])
def test_ternary_exact_per_expert(T, H, E, ld):
    d = gi.dbias_input(T, H, E, seed=21, dist="ternary", ld=ld)
    x = _rows64(d).astype(np.int64)
    o = d.offs.numpy()
    exact = np.stack([x[o[e]:o[e + 1]].sum(axis=0) for e in range(E)])
    assert_bits_equal(_run(d), exact.astype(np.float32), "ternary dbias")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 16, 128])
def test_equals_column_sum_of_each_expert_slice(dtype, W):
    # the column sum oracle is pinned on its own; an expert's dbias is that
    # sum over the expert's rows alone (tiles from the slice's first row)
    d = gi.dbias_input(4000, 24, 5, seed=22, dtype=dtype, ld=32, counts=[1000, 0, 1, 2743, 256])
    got = _run(d, tile_rows=W)
    flat = _flat(d)
    o = d.offs.numpy()
    for e in range(d.E):
        want = np.zeros(d.H, np.float32)
        rows = int(o[e + 1] - o[e])
        oracle.ordered_colsum(flat[o[e] * d.ld:], 1, rows, d.H, rows * d.ld, d.ld, want, tile_rows=W)
        assert_bits_equal(got[e], want, f"expert {e} W={W}")


def test_fp64_bound():
    d = gi.dbias_input(20000, 16, 6, seed=23, dtype=torch.float32)
    x = _rows64(d)
    o = d.offs.numpy()
    got = _run(d).astype(np.float64)
    for e in range(d.E):
        seg = x[o[e]:o[e + 1]]
        exact = seg.sum(axis=0)
        k = int(math.log2(128)) + -(-seg.shape[0] // 128)
        assert np.all(np.abs(got[e] - exact) <= gamma(k) * np.abs(seg).sum(axis=0))
        assert rel_l2(got[e], exact) <= 1e-5


def test_tiles_start_at_each_expert():
    # W = 2, expert 1 owns rows 1..3 = (2^24, 1, 1). Tiles from its first row:
    # (2^24 + 1 -> 2^24) then + 1 -> 2^24 (ties to even, both times). Tiles
    # counted from row 0 would pair rows (2, 3) first: 2^24 + 2, exact.
    col = np.array([5.0, 2.0 ** 24, 1.0, 1.0], np.float32)
    d = gi.DbiasInput(torch.from_numpy(col.reshape(4, 1)), torch.tensor([0, 1, 4]),
                      torch.zeros(2, 1), 4, 1, 1, 2)
    got = _run(d, tile_rows=2)
    assert got[0, 0] == np.float32(5.0)
    assert got[1, 0] == np.float32(2.0 ** 24)


def test_accumulate_is_one_rounding_and_empty_experts():
    # expert 0: rows (1, 1) in two W = 1 tiles: F = 2; out0 = 2^24 -> 2^24 + 2
    # (exact). Adding the partials into out one by one would give 2^24.
    col = np.array([1.0, 1.0], np.float32)
    d = gi.DbiasInput(torch.from_numpy(col.reshape(2, 1)), torch.tensor([0, 2, 2]),
                      torch.zeros(2, 1), 2, 1, 1, 2)
    out0 = np.array([[2.0 ** 24], [-3.5]], np.float32)
    got = _run(d, out0, accumulate=True, tile_rows=1)
    assert got[0, 0] == np.float32(2.0 ** 24 + 2)
    assert got[1, 0] == np.float32(-3.5)          # empty expert: untouched
    got = _run(d, out0, tile_rows=1)
    assert got[1, 0] == 0.0 and not np.signbit(got[1, 0])  # empty expert: +0.0 on overwrite


def test_strided_rows_skip_poison():
    d = gi.dbias_input(3000, 24, 3, seed=24, ld=40)
    got = _run(d)
    assert np.all(np.isfinite(got))
    dense = gi.DbiasInput(d.dY[:, :24].contiguous(), d.offs, d.out, d.T, 24, 24, d.E)
    assert_bits_equal(got, _run(dense), "strided vs compact")


def test_rejects_offsets_outside_the_contract():
    d = gi.dbias_input(100, 8, 2, seed=25)
    out = np.zeros(16, np.float32)
    for bad in ([0, 60, 50], [1, 50, 100], [0, 50, 99]):
        with pytest.raises(ValueError):
            oracle.grouped_dbias(_flat(d), 100, 8, 8, np.array(bad), out)
