"""GPU parity of the aux-loss scalar against the CPU oracle (bit-exact).

Megatron-LM PR #7441, Source 5: the router aux loss summed in the canonical
order (each token's row dot with the expert counts, then the column sum over
tokens) instead of a cross-block float atomicAdd. Cases: ragged token tiles,
expert counts that are not a multiple of 4 (scalar loads) or span several
expert tiles, strided rows, one token, no tokens; the 65536 x 128 workload
with 20 replays under side-stream contention.
"""
import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from gpu_util import assert_replays_identical

pytestmark = pytest.mark.gpu


def _gpu(probs: torch.Tensor, tpe: torch.Tensor, scale: float) -> np.float32:
    return dgr.aux_loss(probs.cuda(), tpe.cuda(), scale).cpu().numpy()[0]


@pytest.mark.parametrize("N,E", [(5000, 128), (4097, 64), (3000, 300), (1000, 7), (129, 1024), (1, 128),
                                 (200, 130)])
def test_parity(N, E):
    a = gi.aux_input(N, E, seed=800 + N + E)
    want = oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), a.scale)
    got = _gpu(a.probs, a.tpe, a.scale)
    assert got.view(np.uint32) == want.view(np.uint32), (got, want)


def test_strided_rows_and_no_tokens():
    a = gi.aux_input(3000, 60, seed=83)
    wide = torch.full((3000, 68), float("nan"))
    wide[:, :60] = a.probs
    want = oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), a.scale)
    got = dgr.aux_loss(wide.cuda()[:, :60], a.tpe.cuda(), a.scale).cpu().numpy()[0]
    assert got.view(np.uint32) == want.view(np.uint32)
    z = dgr.aux_loss(torch.zeros((0, 8), device="cuda"), torch.ones(8, dtype=torch.int32, device="cuda"), -2.0)
    assert z.cpu().numpy()[0].view(np.uint32) == np.float32(-2.0 * 0.0).view(np.uint32)


def test_full_workload_and_replays():
    a = gi.aux_full()
    probs, tpe = a.probs.cuda(), a.tpe.cuda()
    out = torch.empty(1, device="cuda")
    ws = dgr.workspace(dgr.aux_loss_workspace_bytes(probs.shape[0]))
    got = assert_replays_identical(lambda: dgr.aux_loss(probs, tpe, a.scale, out, ws=ws), n=20)
    want = oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), a.scale)
    assert got.view(np.float32)[0].view(np.uint32) == want.view(np.uint32)
