"""GPU parity of the grouped dbias against the CPU oracle (bit-exact).

cuDNN-frontend PR #521, commit "Cover dbias": per-expert ordered column sums
of dY with device offsets. Small cases span several tiles per expert, ragged
last tiles, empty experts, every tile width, bf16 and fp32, strided rows with
NaN poison past H and column blocks that end inside H; the 65536 x 2048
workload (8 experts) runs at full size with 20 replays under side-stream
contention; offsets outside the contract are refused on the device.
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


def _flat(d: gi.DbiasInput) -> np.ndarray:
    return gi.bits(d.dY).reshape(-1) if d.dY.dtype == torch.bfloat16 else gi.f32(d.dY).reshape(-1)


def _oracle(d: gi.DbiasInput, W=128, accumulate=False) -> np.ndarray:
    out = gi.f32(d.out).reshape(-1).copy()
    oracle.grouped_dbias(_flat(d), d.T, d.H, d.ld, d.offs.numpy(), out, accumulate=accumulate, tile_rows=W)
    return out.reshape(d.E, d.H)


def _gpu(d: gi.DbiasInput, W=128, accumulate=False, ws=None, dev=None) -> torch.Tensor:
    dY, offs, out0 = (d.dY.cuda(), d.offs.cuda(), d.out.cuda()) if dev is None else dev
    out = out0.clone()
    dgr.grouped_dbias(dY[:, :d.H], offs, out, accumulate=accumulate, tile_rows=W, ws=ws)
    return out


CASES = [
    # T, H, E, dtype, W, ld, counts, accumulate
    (5000, 64, 4, torch.bfloat16, 128, None, None, False),
    (5000, 64, 4, torch.bfloat16, 128, None, None, True),
    (3001, 24, 3, torch.bfloat16, 128, 40, None, False),      # strided rows, one short column block
    (4000, 520, 5, torch.bfloat16, 128, None, [1000, 0, 1, 2743, 256], True),   # empty and 1-row experts
    (4000, 520, 5, torch.bfloat16, 128, None, [1000, 0, 1, 2743, 256], False),
    (2500, 36, 2, torch.float32, 128, 44, None, False),       # fp32 rows
    (2500, 300, 6, torch.float32, 64, None, None, True),
    (1000, 16, 3, torch.bfloat16, 8, None, None, False),      # every tile width
    (1000, 16, 3, torch.bfloat16, 16, None, None, False),
    (1000, 16, 3, torch.bfloat16, 32, None, None, False),
    (1, 8, 1, torch.bfloat16, 128, None, None, False),        # one row
    (700, 8, 64, torch.bfloat16, 128, None, None, False),     # many experts, most tiny or empty
    (9000, 2048, 300, torch.bfloat16, 128, None, None, True),  # experts across two prefix passes
]


@pytest.mark.parametrize("T,H,E,dtype,W,ld,counts,acc", CASES)
def test_parity_small(T, H, E, dtype, W, ld, counts, acc):
    d = gi.dbias_input(T, H, E, seed=600 + T + H + E + W, dtype=dtype, ld=ld, counts=counts,
                       out_init="random" if acc else "zeros")
    want = _oracle(d, W, acc)
    got = _gpu(d, W, acc).cpu().numpy()
    assert_bits_equal(got, want, f"dbias T={T} H={H} E={E} W={W} acc={acc}")


def test_overwrite_zeroes_empty_experts_and_accumulate_leaves_them():
    d = gi.dbias_input(3000, 64, 4, seed=31, counts=[0, 3000, 0, 0], out_init="random")
    got = _gpu(d).cpu().numpy()
    assert not np.any(got[[0, 2, 3]]) and not np.any(np.signbit(got[[0, 2, 3]]))
    got = _gpu(d, accumulate=True).cpu().numpy()
    assert_bits_equal(got[[0, 2, 3]], gi.f32(d.out)[[0, 2, 3]], "empty experts untouched")


def test_full_workload_and_replays():
    d = gi.dbias_full()
    want = _oracle(d)
    dev = (d.dY.cuda(), d.offs.cuda(), d.out.cuda())
    ws = dgr.workspace(dgr.dbias_workspace_bytes(d.T, d.H, d.E))
    got = assert_replays_identical(lambda: _gpu(d, dev=dev, ws=ws), n=20)
    assert_bits_equal(got.view(np.float32), want, "dbias 65536 x 2048")
    assert dgr.read_device_status(ws) == 0


def test_offsets_outside_the_contract_are_refused_on_the_device():
    d = gi.dbias_input(1000, 16, 2, seed=32)
    dY = d.dY.cuda()
    for bad in ([0, 600, 500], [1, 500, 1000], [0, 500, 999]):
        ws = dgr.workspace(dgr.dbias_workspace_bytes(1000, 16, 2))
        out = torch.full((2, 16), 7.0, device="cuda")
        dgr.grouped_dbias(dY, torch.tensor(bad, device="cuda"), out, ws=ws)
        assert dgr.read_device_status(ws) == 1  # DGR_ERR_INVALID_ARG
        assert torch.all(out == 7.0)
