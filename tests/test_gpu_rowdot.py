"""GPU parity of the ordered dprob against the CPU oracle (bit-exact).

cuDNN-frontend PR #521, commit "deterministic dprob": one slot per N-tile,
reduced in a fixed order and accumulated into dprob. Small cases span several
tiles and ragged ends (vector and scalar paths, bf16 and fp32, leading
dimensions with NaN poison), the slots output, accumulate, the empty cases,
and the 65536 x 4096 workload at full size with 20 replays under contention.
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


def _oracle(di: gi.DprobInput, out0=None, accumulate=False, slots=False):
    fl = gi.bits if di.dY.dtype == torch.bfloat16 else gi.f32
    out = np.zeros(di.M, np.float32) if out0 is None else out0.copy()
    ld = di.dY.shape[1]
    sl = oracle.ordered_rowdot_dprob(fl(di.dY).reshape(-1), fl(di.Y).reshape(-1), di.M, di.N, ld, ld, out,
                                     accumulate=accumulate, return_slots=slots)
    return out, sl


def _gpu(di: gi.DprobInput, out0=None, accumulate=False, slots=None, dev=None):
    dY, Y = (di.dY.cuda(), di.Y.cuda()) if dev is None else dev
    out = torch.zeros(di.M, device="cuda") if out0 is None else torch.from_numpy(out0.copy()).cuda()
    dgr.ordered_rowdot_dprob(dY[:, :di.N], Y[:, :di.N], out, accumulate=accumulate, slots=slots)
    return out


CASES = [
    (64, 4096, None, torch.bfloat16),
    (37, 1000, None, torch.bfloat16),     # ragged tile
    (16, 300, 512, torch.bfloat16),       # leading dimension, poison past N
    (8, 77, 80, torch.bfloat16),          # 16-byte rows (ld 80), ragged vector
    (5, 75, 75, torch.bfloat16),          # unaligned rows: scalar path
    (33, 2000, None, torch.float32),
    (3, 4100, 4104, torch.float32),
    (1, 1, None, torch.bfloat16),
    (1000, 128, None, torch.bfloat16),
    (4, 65536, None, torch.bfloat16),     # the N limit
]


@pytest.mark.parametrize("M,N,ld,dtype", CASES)
def test_parity_small(M, N, ld, dtype):
    di = gi.dprob_input(M, N, seed=300 + M + N, ld=ld, dtype=dtype)
    want, _ = _oracle(di)
    assert_bits_equal(_gpu(di).cpu().numpy(), want, f"dprob {M}x{N} ld={ld}")


def test_slots_and_accumulate():
    di = gi.dprob_input(50, 1000, seed=31)
    out0 = np.random.default_rng(2).standard_normal(50).astype(np.float32)
    want, want_slots = _oracle(di, out0=out0, accumulate=True, slots=True)
    slots = torch.full((50, 8), float("nan"), device="cuda")
    got = _gpu(di, out0=out0, accumulate=True, slots=slots)
    assert_bits_equal(got.cpu().numpy(), want, "accumulate")
    assert_bits_equal(slots.cpu().numpy(), want_slots, "slots")


def test_empty():
    dY = torch.zeros((8, 0), dtype=torch.bfloat16, device="cuda")
    out = torch.full((8,), 3.0, device="cuda")
    dgr.ordered_rowdot_dprob(dY, dY, out)
    assert_bits_equal(out.cpu().numpy(), np.zeros(8, np.float32), "N=0 overwrite")
    out.fill_(3.0)
    dgr.ordered_rowdot_dprob(dY, dY, out, accumulate=True)
    assert_bits_equal(out.cpu().numpy(), np.full(8, 3.0, np.float32), "N=0 accumulate")


def test_full_workload():
    di = gi.dprob_full()
    want, _ = _oracle(di)
    dev = (di.dY.cuda(), di.Y.cuda())
    got = assert_replays_identical(lambda: _gpu(di, dev=dev), n=20)
    assert_bits_equal(got.view(np.float32), want, "dprob 65536x4096")
