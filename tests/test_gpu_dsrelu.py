"""GPU parity of dprob fused into the grouped dsReLU GEMM against the CPU oracle (bit-exact).

cuDNN-frontend PR #521: the GEMM C = A_e B_e is recomputed on the tensor cores
(never written), relu(C)^2 is multiplied by dY, and each (token, N-tile) gets
one partial, folded in order into dprob. The oracle models each K16
tensor-core step bit for bit (pinned against the hardware on its own), so the
comparison is exact. Small cases cover an empty expert, row blocks that end
inside an expert, several k stages and column blocks, accumulate; the 16384 x
2048 x 4096 workload runs at full size, checked on sampled rows, with 20
replays (every other one under side-stream contention); offsets outside the contract are refused.
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


def _oracle(d: gi.DsreluInput, accumulate=False, rows=None):
    out = d.dprob.numpy().copy() if rows is None else d.dprob.numpy()[rows].copy()
    oracle.dsrelu_dprob(gi.bits(d.A), gi.bits(d.B), d.offs.numpy(), gi.bits(d.dY), out, accumulate=accumulate,
                        rows=rows)
    return out


def _gpu(d: gi.DsreluInput, accumulate=False, dev=None, ws=None):
    A, B, offs, dY, dp0 = (d.A.cuda(), d.B.cuda(), d.offs.cuda(), d.dY.cuda(), d.dprob.cuda()) if dev is None else dev
    dp = dp0.clone()
    dgr.dsrelu_dprob(A, B, offs, dY, dp, accumulate=accumulate, ws=ws)
    return dp


CASES = [
    # counts, K, N, accumulate
    ([300, 0, 213], 128, 512, False),
    ([129, 127], 256, 256, False),
    ([1, 200, 64, 5], 64, 768, True),
    ([128], 192, 256, True),
]


@pytest.mark.parametrize("counts,K,N,acc", CASES)
def test_parity(counts, K, N, acc):
    d = gi.dsrelu_input(len(counts), sum(counts), K, N, seed=930 + K + N, counts=counts,
                        out_init="random" if acc else "zeros")
    want = _oracle(d, acc)
    got = _gpu(d, acc).cpu().numpy()
    assert_bits_equal(got, want, f"dsrelu dprob counts={counts} K={K} N={N}")


def test_full_workload_sampled_rows_and_replays():
    d = gi.dsrelu_full()
    dev = (d.A.cuda(), d.B.cuda(), d.offs.cuda(), d.dY.cuda(), d.dprob.cuda())
    ws = dgr.workspace(dgr.dsrelu_dprob_workspace_bytes(16384, 4096))
    got = assert_replays_identical(lambda: _gpu(d, dev=dev, ws=ws), n=20).view(np.float32)
    o = d.offs.numpy()
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([o[:-1], o[1:] - 1, rng.integers(0, 16384, 8)]))
    want = _oracle(d, rows=rows)
    assert_bits_equal(got[rows], want, "dsrelu dprob 16384 x 2048 x 4096 (sampled rows)")
    assert dgr.read_device_status(ws) == 0


def test_offsets_outside_the_contract_are_refused_on_the_device():
    d = gi.dsrelu_input(2, 256, 64, 256, seed=94, counts=[128, 128])
    A, B, dY = d.A.cuda(), d.B.cuda(), d.dY.cuda()
    for bad in ([0, 200, 100], [0, 128, 255]):
        ws = dgr.workspace(dgr.dsrelu_dprob_workspace_bytes(256, 256))
        dp = torch.full((256,), 5.0, device="cuda")
        dgr.dsrelu_dprob(A, B, torch.tensor(bad, device="cuda"), dY, dp, ws=ws)
        assert dgr.read_device_status(ws) == 1
        assert torch.all(dp == 5.0)


def test_no_tokens():
    """Every expert empty (T = 0): nothing to compute; the call succeeds with an empty dprob."""
    d = gi.dsrelu_input(3, 0, 64, 256, seed=78, counts=[0, 0, 0])
    dp = _gpu(d)
    assert dp.numel() == 0
    torch.cuda.synchronize()
