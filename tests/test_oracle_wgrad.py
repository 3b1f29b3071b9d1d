"""Pins of the oracle's grouped weight gradient (FlashInfer PRs #8602 / #8924).

Independent checks: on ternary inputs every product, chunk partial and fold is
an exact integer, so the result must equal numpy's int64 G_e^T X_e plus
main_grad for any arithmetic inside a tensor-core step (this pins the data
flow: expert offsets, chunking, zero-filled tails, the transposition, the
final add); empty experts leave main_grad bitwise unchanged; fp64 within the
error bound; and the K16 step model's own properties (a lone product is exact,
integer sums are exact, the truncation error stays inside its bound).
"""
import numpy as np
import pytest
import torch

import dgr_inputs as gi
import oracle
from util import assert_bits_equal, bf16_bits_to_f64, rel_l2


def _run(wi: gi.WgradInput, chunk=512, sequential=False):
    T, N = wi.G.shape
    K = wi.X.shape[1]
    mg = gi.f32(wi.main_grad).copy()
    oracle.grouped_wgrad_accumulate(gi.bits(wi.G), gi.bits(wi.X), wi.offs.numpy(), wi.E, N, K, mg,
                                    chunk_tokens=chunk, sequential_into_out=sequential)
    return mg


def _exact(wi: gi.WgradInput, dtype=np.int64):
    G = wi.G.to(torch.float64).numpy()
    X = wi.X.to(torch.float64).numpy()
    out = wi.main_grad.to(torch.float64).numpy().copy()
    o = wi.offs.numpy()
    for e in range(wi.E):
        out[e] += G[o[e]:o[e + 1]].T @ X[o[e]:o[e + 1]]
    return out


@pytest.mark.parametrize("counts,chunk", [([700, 0, 1029, 300], 512), ([1, 17, 511, 513], 512),
                                          ([64, 64, 64, 64], 64)])
def test_ternary_exact(counts, chunk):
    wi = gi.wgrad_input(4, sum(counts), 24, 40, seed=41, dist="ternary", counts=counts)
    got = _run(wi, chunk)
    assert_bits_equal(got, _exact(wi).astype(np.float32), "ternary wgrad")


def test_empty_expert_bitwise_unchanged():
    wi = gi.wgrad_input(3, 600, 16, 16, seed=42, counts=[300, 0, 300])
    got = _run(wi)
    assert_bits_equal(got[1], gi.f32(wi.main_grad)[1], "empty expert")
    assert not np.array_equal(got[0], gi.f32(wi.main_grad)[0])


def test_fp64_bound():
    wi = gi.wgrad_input(2, 1500, 16, 24, seed=43, counts=[1100, 400])
    got = _run(wi).astype(np.float64)
    exact = _exact(wi)
    G = np.abs(wi.G.to(torch.float64).numpy())
    X = np.abs(wi.X.to(torch.float64).numpy())
    o = wi.offs.numpy()
    absdot = np.stack([G[o[e]:o[e + 1]].T @ X[o[e]:o[e + 1]] for e in range(2)])
    absdot += np.abs(wi.main_grad.numpy())
    # per K16 step at most 17 terms truncated at 2^-(frac_bits) of the step's
    # largest term, plus one fp32 rounding; 32 steps, 3 folds, one final add
    bound = 64 * 2.0 ** -22 * absdot
    assert np.all(np.abs(got - exact) <= bound)
    assert rel_l2(got, exact) <= 1e-5


def test_elements_match_full_and_fold_differs_from_sequential():
    wi = gi.wgrad_input(2, 2000, 8, 8, seed=44, counts=[1500, 500])
    full = _run(wi)
    e = np.array([0, 0, 1, 1]); n = np.array([0, 7, 3, 5]); k = np.array([0, 7, 1, 2])
    mg = gi.f32(wi.main_grad)[e, n, k]
    res = oracle.wgrad_elements(gi.bits(wi.G), gi.bits(wi.X), wi.offs.numpy(), 8, 8, e, n, k, mg)
    assert_bits_equal(res, full[e, n, k], "elements vs full")
    seq = _run(wi, sequential=True)
    assert not np.array_equal(full.view(np.uint32), seq.view(np.uint32))


def _bf16(vals):
    return (torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
            .view(torch.int16).numpy().view(np.uint16))


def test_k16_lone_product_is_exact():
    rng = np.random.default_rng(6)
    a = np.zeros((1000, 16), np.uint16); b = np.zeros((1000, 16), np.uint16)
    lane = rng.integers(0, 16, 1000)
    av = _bf16(rng.standard_normal(1000)); bv = _bf16(rng.standard_normal(1000))
    a[np.arange(1000), lane] = av; b[np.arange(1000), lane] = bv
    res = oracle.tc_k16_batch(np.zeros(1000, np.float32), np.zeros(1000, np.int32), a, b)
    want = (bf16_bits_to_f64(av) * bf16_bits_to_f64(bv)).astype(np.float32)
    assert_bits_equal(res, want, "lone product")


def test_k16_integer_sums_exact_and_bound_on_random():
    rng = np.random.default_rng(7)
    n = 20000
    ai = rng.integers(-100, 101, (n, 16)); bi = rng.integers(-100, 101, (n, 16))
    acc = rng.integers(-10 ** 6, 10 ** 6, n).astype(np.float32)
    res = oracle.tc_k16_batch(acc, np.ones(n, np.int32), _bf16(ai), _bf16(bi))
    assert_bits_equal(res, (acc.astype(np.int64) + (ai * bi).sum(1)).astype(np.float32), "integers")
    # random data: the model stays within its truncation bound of the exact sum
    a = _bf16(rng.standard_normal((n, 16))); b = _bf16(rng.standard_normal((n, 16)))
    acc = rng.standard_normal(n).astype(np.float32)
    res = oracle.tc_k16_batch(acc, np.ones(n, np.int32), a, b).astype(np.float64)
    p = bf16_bits_to_f64(a) * bf16_bits_to_f64(b)
    exact = acc.astype(np.float64) + p.sum(1)
    biggest = np.maximum(np.abs(p).max(1), np.abs(acc))
    assert np.all(np.abs(res - exact) <= 18 * 2.0 ** -23 * biggest * 2)
