"""GPU parity of the ordered column sum against the CPU oracle (bit-exact).

Megatron-LM PR #8244, description: FP32 partials per program, reduced by the
caller in order. Every output is compared bit for bit with the oracle on the
same seeded host bytes: small cases that span several tiles and a ragged tail
(vector and scalar load paths, bf16 and fp32, strided views, every tile
width), the three workloads at full size, 20 replays under side-stream
contention, workspace reuse and the empty cases.
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


def _oracle(ci: gi.ColsumInput, W=128, out0=None, accumulate=False):
    flat = gi.bits(ci.base) if ci.base.dtype == torch.bfloat16 else gi.f32(ci.base)
    out = np.zeros(ci.H, np.float32) if out0 is None else out0.copy()
    oracle.ordered_colsum(flat, ci.B, ci.S, ci.H, ci.stride_b, ci.stride_s, out, accumulate=accumulate,
                          tile_rows=W)
    return out


def _view(ci: gi.ColsumInput, base_dev: torch.Tensor) -> torch.Tensor:
    return base_dev.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))


def _gpu(ci: gi.ColsumInput, W=128, out0=None, accumulate=False, ws=None, base_dev=None):
    base_dev = ci.base.cuda() if base_dev is None else base_dev
    out = torch.zeros(ci.H, device="cuda") if out0 is None else torch.from_numpy(out0.copy()).cuda()
    dgr.ordered_colsum(_view(ci, base_dev), out, accumulate=accumulate, tile_rows=W, ws=ws)
    return out


CASES = [
    # B, S, H, token_stride, dtype, W
    (1, 2048, 16, None, torch.bfloat16, 128),
    (1, 1000, 16, None, torch.bfloat16, 128),    # ragged last tile
    (3, 333, 64, 128, torch.bfloat16, 128),      # strided, tiles cross batches
    (2, 700, 12, None, torch.bfloat16, 128),     # H % 8 != 0: scalar loads
    (1, 5000, 40, None, torch.float32, 128),     # fp32 vector path
    (2, 999, 7, 9, torch.float32, 64),           # fp32 scalar path
    (1, 4097, 64, None, torch.bfloat16, 1),      # sequential tiles
    (1, 3000, 64, None, torch.bfloat16, 32),
    (1, 9000, 24, None, torch.bfloat16, 4096),
    (1, 100, 16, None, torch.bfloat16, 256),     # one partial tile
    (1, 1, 8, None, torch.bfloat16, 128),
    (1, 70000, 520, None, torch.bfloat16, 128),  # several column blocks and folders
    (1, 3000, 4096, None, torch.bfloat16, 128),  # the H limit
    # warp producers: up to 512 tiles one launch with a ticket, beyond it folders
    (1, 65536, 64, None, torch.bfloat16, 128),   # 512 tiles: the ticket path's largest
    (1, 65537, 64, None, torch.bfloat16, 128),   # 513 tiles: warp producers and folders
    (4, 16, 8, 24, torch.bfloat16, 128),         # ticket path, strided, one tile across batches
    (1, 100000, 64, None, torch.bfloat16, 128),  # ragged last tile
    (3, 40000, 16, None, torch.bfloat16, 128),
    (1, 50000, 32, None, torch.float32, 128),
    (1, 60000, 64, None, torch.bfloat16, 64),
    (1, 20001, 8, None, torch.bfloat16, 16),
]


@pytest.mark.parametrize("B,S,H,ts,dtype,W", CASES)
def test_parity_small(B, S, H, ts, dtype, W):
    ci = gi.colsum_input(B, S, H, seed=100 + S + H, token_stride=ts, dtype=dtype)
    assert_bits_equal(_gpu(ci, W).cpu().numpy(), _oracle(ci, W), f"colsum {B}x{S}x{H} W={W}")


def test_accumulate_and_reuse_of_workspace():
    ci = gi.colsum_input(2, 3000, 64, seed=7)
    ws = dgr.workspace(dgr.colsum_workspace_bytes(6000, 64))
    out0 = np.random.default_rng(1).standard_normal(64).astype(np.float32)
    want = _oracle(ci, out0=out0, accumulate=True)
    base = ci.base.cuda()
    for _ in range(3):  # the same workspace, reused: counters must come back to zero
        got = _gpu(ci, out0=out0, accumulate=True, ws=ws, base_dev=base)
        assert_bits_equal(got.cpu().numpy(), want, "accumulate")
    assert dgr.read_device_status(ws) == 0


def test_empty():
    out = torch.full((16,), 5.0, device="cuda")
    x = torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda")
    dgr.ordered_colsum(x, out)
    assert_bits_equal(out.cpu().numpy(), np.zeros(16, np.float32), "T=0 overwrite")
    out.fill_(5.0)
    dgr.ordered_colsum(x, out, accumulate=True)
    assert_bits_equal(out.cpu().numpy(), np.full(16, 5.0, np.float32), "T=0 accumulate")


@pytest.mark.parametrize("name", ["colsum_small", "colsum_strided"])
def test_full_workloads_small(name):
    ci = getattr(gi, name)()
    want = _oracle(ci)
    assert np.all(np.isfinite(want))
    base = ci.base.cuda()
    got = assert_replays_identical(lambda: _gpu(ci, base_dev=base), n=20)
    assert_bits_equal(got.view(np.float32), want, name)


def test_full_workload_large():
    ci = gi.colsum_large()
    want = _oracle(ci)
    base = ci.base.cuda()
    ws = dgr.workspace(dgr.colsum_workspace_bytes(ci.B * ci.S, ci.H))
    got = assert_replays_identical(lambda: _gpu(ci, base_dev=base, ws=ws), n=20)
    assert_bits_equal(got.view(np.float32), want, "colsum_large")
    assert dgr.read_device_status(ws) == 0


@pytest.mark.parametrize("S,H,W", [
    (600 * 128 + 1, 32, 128),  # warp producers and folders; the last tile is one row
    (3001, 12, 1),             # block producers (3 vectors a row), one-row tiles
    (200 * 128 + 1, 32, 128),  # one launch with a ticket
])
def test_nan_partial_and_workspace_back_to_zero(S, H, W):
    # A slot word holds the complement of a tile partial, 0 meaning "not
    # written yet"; the NaN with every bit set (complement 0) is stored as
    # another NaN. Here it is a whole tile's partial (a one-row tile): its
    # column must come out NaN, every other column bit-exact, and every word
    # of the workspace must be zero again after each call.
    ci = gi.colsum_input(1, S, H, seed=S + H, dtype=torch.float32)
    ci.base.view(torch.int32)[(S - 1) * H + 3] = -1
    want = _oracle(ci, W)
    assert np.isnan(want[3])
    keep = np.arange(H) != 3
    ws = dgr.workspace(dgr.colsum_workspace_bytes(S, H, W))
    base = ci.base.cuda()
    for _ in range(2):
        got = _gpu(ci, W, ws=ws, base_dev=base).cpu().numpy()
        assert np.isnan(got[3])
        assert_bits_equal(got[keep], want[keep], f"colsum {S}x{H} W={W} beside a NaN column")
        assert int(torch.count_nonzero(ws)) == 0
