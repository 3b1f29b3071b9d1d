"""Pins of the oracle's ordered column sum (Megatron-LM PR #8244, description).

Independent checks: exact integer sums (ternary inputs make every partial an
integer below 2^24, so every order gives the exact int64 sum), the fp64 sum
within a relative L2 of 1e-5 and within the elementwise pairwise
error bound, the sequential special case, stride handling against a compacted
copy with NaN poison in the gaps, and the accumulate/empty conventions.
"""
import math

import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal, bf16_bits_to_f64, gamma, rel_l2


def _flat(ci: gi.ColsumInput) -> np.ndarray:
    return gi.bits(ci.base) if ci.base.dtype == torch.bfloat16 else gi.f32(ci.base)


def _dense64(ci: gi.ColsumInput) -> np.ndarray:
    """x as fp64 [T, H], read through the strides."""
    rows = []
    for b in range(ci.B):
        blk = ci.base[b * ci.stride_b: b * ci.stride_b + ci.S * ci.stride_s].view(ci.S, ci.stride_s)
        rows.append(blk[:, :ci.H].to(torch.float64))
    return torch.cat(rows).numpy()


def _run(ci, **kw):
    out = np.zeros(ci.H, np.float32)
    oracle.ordered_colsum(_flat(ci), ci.B, ci.S, ci.H, ci.stride_b, ci.stride_s, out, **kw)
    return out


@pytest.mark.parametrize("B,S,H,ts", [(1, 2048, 16, None), (4, 2048, 64, 128), (3, 1000, 24, 40),
                                      (2, 129, 8, None)])
def test_ternary_exact(B, S, H, ts):
    ci = gi.colsum_input(B, S, H, seed=11, dist="ternary", token_stride=ts)
    exact = _dense64(ci).astype(np.int64).sum(axis=0)
    got = _run(ci)
    assert_bits_equal(got, exact.astype(np.float32), "ternary colsum")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 32, 128, 256])
def test_fp64_bound(dtype, W):
    ci = gi.colsum_input(2, 3000, 16, seed=12, dist="normal", dtype=dtype)
    x = _dense64(ci)
    exact = x.sum(axis=0)
    got = _run(ci, tile_rows=W).astype(np.float64)
    T = ci.B * ci.S
    k = int(math.log2(W)) + -(-T // W)
    bound = gamma(k) * np.abs(x).sum(axis=0)
    assert np.all(np.abs(got - exact) <= bound)
    assert rel_l2(got, exact) <= 1e-5


def test_small_workload_fp64():
    ci = gi.colsum_small()
    x = _dense64(ci)
    got = _run(ci)
    assert rel_l2(got, x.sum(axis=0)) <= 1e-5


def test_strided_view_equals_compacted_copy_and_skips_poison():
    ci = gi.colsum_input(4, 512, 64, seed=13, token_stride=128)
    got = _run(ci)
    assert np.all(np.isfinite(got))
    dense = ci.base.view(4, 512, 128)[..., :64].contiguous().reshape(-1)
    cc = gi.ColsumInput(dense, 4, 512, 64, 512 * 64, 64)
    assert_bits_equal(got, _run(cc), "strided vs compact")


def test_tiles_cross_batch_boundaries_in_flat_token_order():
    # S = 100 is not a multiple of the tile: tokens are flattened t = b*S + s,
    # so a [B, S] input equals the same tokens laid out as [1, B*S]
    ci = gi.colsum_input(5, 100, 8, seed=14)
    flat = gi.ColsumInput(ci.base, 1, 500, 8, 500 * 8, 8)
    assert_bits_equal(_run(ci, tile_rows=64), _run(flat, tile_rows=64), "batch flattening")


def test_slots_and_fold():
    ci = gi.colsum_input(1, 1000, 16, seed=15)
    out = np.zeros(16, np.float32)
    slots = oracle.ordered_colsum(gi.bits(ci.base), 1, 1000, 16, 1000 * 16, 16, out,
                                  return_slots=True)
    assert slots.shape == (8, 16)
    # slot j is the pairwise partial of its own tile; the output folds them in order
    x = bf16_bits_to_f64(gi.bits(ci.base)).reshape(1000, 16).astype(np.float32)
    for j in (0, 7):
        rows = x[j * 128:(j + 1) * 128]
        for h in (0, 15):
            assert_bits_equal(slots[j, h], oracle.pairwise(rows[:, h], 128))
    for h in range(16):
        assert_bits_equal(out[h], oracle.fold(slots[:, h]))


def test_accumulate_is_one_rounding_on_top_of_overwrite():
    ci = gi.colsum_input(1, 777, 16, seed=16)
    fresh = _run(ci)
    rng = np.random.default_rng(4)
    out0 = rng.standard_normal(16).astype(np.float32) * 100
    out = out0.copy()
    oracle.ordered_colsum(_flat(ci), 1, 777, 16, 777 * 16, 16, out, accumulate=True)
    assert_bits_equal(out, (out0 + fresh).astype(np.float32), "accumulate")


def test_empty_input():
    x = np.zeros(1, np.uint16)
    out = np.full(4, -5.0, np.float32)
    oracle.ordered_colsum(x, 0, 10, 4, 40, 4, out)
    assert_bits_equal(out, np.zeros(4, np.float32), "T=0 overwrite gives +0.0")
    out = np.full(4, -5.0, np.float32)
    oracle.ordered_colsum(x, 3, 0, 4, 0, 4, out, accumulate=True)
    assert_bits_equal(out, np.full(4, -5.0, np.float32), "T=0 accumulate leaves out")
