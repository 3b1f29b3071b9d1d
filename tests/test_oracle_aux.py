"""Pins of the oracle's aux-loss scalar (Megatron-LM PR #7441, Source 5).

The loss is RN(scale * S), S the sum over tokens and experts of
probs * tokens_per_expert in the canonical order: each token's row dot (the
dprob reduction, expert tiles of 128) and then the column sum at H = 1 over
tokens (token tiles of 128). Independent checks: the composition of the two
separately pinned oracles (row dot against a broadcast row of counts, then the
column sum of one column) gives the same bits; ternary probabilities with small
counts give the exact integer sum; the fp64 sum within the error bound; the
empty case.
"""
import math

import numpy as np
import pytest

import dgr_inputs as gi
import oracle
from util import gamma


@pytest.mark.parametrize("N,E", [(5000, 128), (3000, 64), (1000, 300), (127, 8), (1, 1)])
def test_equals_row_dot_then_column_sum(N, E):
    a = gi.aux_input(N, E, seed=80 + E)
    p = a.probs.numpy()
    tpe = a.tpe.numpy()
    x = np.zeros(N, np.float32)
    Y = np.broadcast_to(tpe.astype(np.float32), (N, E)).copy()
    oracle.ordered_rowdot_dprob(p.reshape(-1), Y.reshape(-1), N, E, E, E, x)
    s = np.zeros(1, np.float32)
    oracle.ordered_colsum(x, 1, N, 1, N, 1, s)
    want = np.float32(np.float32(a.scale) * s[0])
    got = oracle.aux_loss(p, tpe, a.scale)
    assert got.view(np.uint32) == want.view(np.uint32)


@pytest.mark.parametrize("N,E", [(65536, 128), (4000, 200)])
def test_ternary_exact(N, E):
    a = gi.aux_input(N, E, seed=81, dist="ternary")
    tpe = (np.arange(E) % 5).astype(np.int32)
    exact = int((a.probs.numpy().astype(np.int64) * tpe.astype(np.int64)).sum())
    assert abs(exact) < 2 ** 24
    assert oracle.aux_loss(a.probs.numpy(), tpe, 1.0) == np.float32(exact)


def test_fp64_bound():
    a = gi.aux_input(20000, 128, seed=82)
    p = a.probs.numpy().astype(np.float64)
    t = a.tpe.numpy().astype(np.float64)
    terms = p * t
    exact = terms.sum()
    got = float(oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), 1.0))
    k = 1 + 7 + 7 + -(-20000 // 128)  # product, expert tree, token tree, token-tile fold
    assert abs(got - exact) <= gamma(k) * np.abs(terms).sum()


def test_empty():
    assert oracle.aux_loss(np.zeros((0, 8), np.float32), np.ones(8, np.int32), 3.0) == 0.0
