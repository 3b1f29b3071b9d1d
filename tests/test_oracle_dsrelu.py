"""Pins of the oracle's dprob fused into the grouped dsReLU GEMM (cuDNN-frontend PR #521).

dprob[m] = fold over N-tiles of pw_128(RN(dY * RN(relu(C)^2))) with C = A_e B_e
by tensor-core K16 steps (the K16 model is pinned against the hardware on its
own). Independent checks: C rebuilt step by step with the K16 model and the
rest through the separately pinned row-dot oracle gives the same bits; ternary
inputs give the exact integer result; a subset of rows equals those rows of
the full computation; accumulate is one rounding; an empty expert is fine.
"""
import numpy as np
import pytest

import dgr_inputs as gi
import oracle


def _bits(t):
    return gi.bits(t)


def _C_by_steps(d: gi.DsreluInput) -> np.ndarray:
    A, B = _bits(d.A), _bits(d.B)
    T, K = A.shape
    E, _, N = B.shape
    o = d.offs.numpy()
    C = np.zeros((T, N), np.float32)
    for e in range(E):
        rows = np.arange(o[e], o[e + 1])
        if rows.size == 0:
            continue
        acc = np.zeros((rows.size, N), np.float32)
        for s in range(K // 16):
            a = np.repeat(A[rows, 16 * s:16 * s + 16][:, None, :], N, axis=1).reshape(-1, 16)
            b = np.tile(B[e, 16 * s:16 * s + 16, :].T, (rows.size, 1))
            has = np.full(a.shape[0], 1 if s > 0 else 0, np.int32)
            acc = oracle.tc_k16_batch(acc.reshape(-1), has, a, b).reshape(rows.size, N)
        C[rows] = acc
    return C


@pytest.mark.parametrize("E,counts,K,N", [(3, [40, 0, 27], 64, 256), (2, [33, 31], 128, 200)])
def test_equals_k16_steps_then_row_dot(E, counts, K, N):
    d = gi.dsrelu_input(E, sum(counts), K, N, seed=90 + K, counts=counts)
    C = _C_by_steps(d)
    r = np.maximum(C, np.float32(0))
    Y = (r * r).astype(np.float32)
    dY = d.dY.float().numpy()
    want = np.zeros(d.A.shape[0], np.float32)
    oracle.ordered_rowdot_dprob(dY.reshape(-1), Y.reshape(-1), dY.shape[0], N, N, N, want)
    got = np.zeros_like(want)
    oracle.dsrelu_dprob(_bits(d.A), _bits(d.B), d.offs.numpy(), _bits(d.dY), got)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_ternary_exact():
    d = gi.dsrelu_input(2, 90, 64, 384, seed=91, dist="ternary", counts=[50, 40])
    A = d.A.double().numpy()
    B = d.B.double().numpy()
    o = d.offs.numpy()
    C = np.concatenate([A[o[e]:o[e + 1]] @ B[e] for e in range(2)])
    exact = (d.dY.double().numpy() * np.maximum(C, 0) ** 2).sum(axis=1)
    assert np.abs(exact).max() < 2 ** 24
    got = np.zeros(90, np.float32)
    oracle.dsrelu_dprob(_bits(d.A), _bits(d.B), o, _bits(d.dY), got)
    assert np.array_equal(got, exact.astype(np.float32))


def test_rows_subset_and_accumulate():
    d = gi.dsrelu_input(3, 120, 64, 256, seed=92, counts=[50, 0, 70], out_init="random")
    full = d.dprob.numpy().copy()
    oracle.dsrelu_dprob(_bits(d.A), _bits(d.B), d.offs.numpy(), _bits(d.dY), full, accumulate=True)
    rows = np.array([0, 49, 50, 119, 77])
    sub = d.dprob.numpy()[rows].copy()
    oracle.dsrelu_dprob(_bits(d.A), _bits(d.B), d.offs.numpy(), _bits(d.dY), sub, accumulate=True, rows=rows)
    assert np.array_equal(sub.view(np.uint32), full[rows].view(np.uint32))
    over = np.zeros(120, np.float32)
    oracle.dsrelu_dprob(_bits(d.A), _bits(d.B), d.offs.numpy(), _bits(d.dY), over)
    assert np.array_equal(full.view(np.uint32), (d.dprob.numpy() + over).view(np.uint32))
