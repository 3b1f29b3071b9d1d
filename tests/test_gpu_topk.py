"""GPU parity of the canonical compact top-K against the CPU oracle.

Megatron-LM PR #7441, Source 1: ids sorted per row (padding last), logits
permuted alike, softmax of the valid slots recomputed in that order. Ids,
permuted logits and probabilities are all bit-exact: kernel and oracle each
compute the exponential by Tang's table-driven method in the same binary32
steps (the oracle's is pinned against exp in binary64 on its own).
Determinism is pinned bit for bit on the GPU itself too: any order of a row's
slots gives the same outputs, and 20 replays under side-stream contention are
identical. K from 1 to 256, padding other than -1, rows that are all padding,
the 65536 x 128 workload.
"""
import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from gpu_util import assert_replays_identical
from util import assert_bits_equal

pytestmark = pytest.mark.gpu


def _gpu(ids: np.ndarray, lg: np.ndarray):
    oi, ol, pr = dgr.topk_canonicalize(torch.from_numpy(ids).cuda(), torch.from_numpy(lg).cuda())
    return oi.cpu().numpy(), ol.cpu().numpy(), pr.cpu().numpy()


def _check(ids, lg, what):
    want = oracle.topk_canonicalize(ids, lg)
    got = _gpu(ids, lg)
    assert np.array_equal(got[0], want[0]), what
    assert_bits_equal(got[1], want[1], what + " logits")
    assert_bits_equal(got[2], want[2], what + " probs")


@pytest.mark.parametrize("R,K", [(1000, 128), (700, 256), (500, 200), (900, 64), (800, 33), (600, 7), (64, 1)])
def test_parity(R, K):
    t = gi.topk_input(R, K, seed=700 + K, n_keys=65536 if K > 1 else 10, pad_row_every=16)
    _check(t.ids.numpy(), t.logits.numpy(), f"topk R={R} K={K}")


@pytest.mark.parametrize("K", [128, 256, 40])
def test_parity_wide_ids(K):
    # ids up to 2^30: rows whose ids do not all fit the 32-bit sort key take
    # the 64-bit one; one row in four keeps small ids (32-bit keys)
    t = gi.topk_input(800, K, seed=750 + K, n_keys=1 << 30)
    ids = t.ids.numpy().copy()
    ids[::4] = np.where(ids[::4] < 0, ids[::4], ids[::4] >> 8)  # unique and below 2^23
    _check(ids, t.logits.numpy(), f"topk wide ids K={K}")


def test_padding_values_and_equal_logits():
    t = gi.topk_input(300, 128, seed=71, pad_frac=0.3)
    ids = t.ids.numpy().copy()
    ids[ids < 0] = -7  # any negative id is padding and comes out unchanged
    lg = t.logits.numpy().copy()
    lg[::3] = 1.25  # equal logits: exactly 1 / n
    _check(ids, lg, "padding -7, equal logits")


def test_slot_order_does_not_matter_on_the_gpu():
    t = gi.topk_input(2000, 128, seed=72)
    ids, lg = t.ids.numpy(), t.logits.numpy()
    ref = _gpu(ids, lg)
    full = ~(ids < 0).any(axis=1)
    rng = np.random.default_rng(9)
    for _ in range(3):
        order = np.argsort(rng.random(ids.shape), axis=1)
        got = _gpu(np.take_along_axis(ids, order, 1), np.take_along_axis(lg, order, 1))
        assert np.array_equal(got[0], ref[0])
        assert_bits_equal(got[1][full], ref[1][full], "logits of rows without padding")
        assert_bits_equal(got[2], ref[2], "probs")


def test_full_workload_and_replays():
    t = gi.topk_full()
    ids, lg = t.ids.cuda(), t.logits.cuda()
    out = (torch.empty_like(ids), torch.empty_like(lg), torch.empty_like(lg))

    def run():
        dgr.topk_canonicalize(ids, lg, *out)
        return out[2]
    probs = assert_replays_identical(run, n=20)
    want = oracle.topk_canonicalize(t.ids.numpy(), t.logits.numpy())
    assert np.array_equal(out[0].cpu().numpy(), want[0])
    assert_bits_equal(out[1].cpu().numpy(), want[1], "topk 65536 x 128 logits")
    assert_bits_equal(probs.view(np.float32), want[2], "topk 65536 x 128 probs")


def test_no_rows():
    """R = 0: nothing to compute; the call succeeds and returns empty outputs."""
    got = _gpu(np.zeros((0, 8), np.int32), np.zeros((0, 8), np.float32))
    assert all(a.shape == (0, 8) for a in got)
