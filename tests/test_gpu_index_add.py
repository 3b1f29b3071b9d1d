"""GPU parity of the deterministic index_add against the CPU oracle (bit-exact).

Megatron-LM PR #7441, Source 3: stable sort by destination plus a segmented
sum, padding routed to the dummy row. Small cases cover every tile width
(1 = sequential .. 128), rows big enough to take the split path, bad indices
and their count, random initial rows (untouched rows keep their bits),
strided rows, several column blocks and the empty cases; the 262144 x 128
workload runs at full size with 20 replays under side-stream contention.
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


def _oracle(ia: gi.IndexAddInput, seg_tile=128):
    out = gi.f32(ia.out).copy()
    src = gi.f32(ia.src)
    N, D = src.shape
    bad, _, _ = oracle.det_index_add(out, ia.R, D, D, src, D, ia.idx.numpy(), N, seg_tile=seg_tile)
    return out, bad


def _gpu(ia: gi.IndexAddInput, seg_tile=128, dev=None, ws=None, bad=None):
    src, idx, out0 = (ia.src.cuda(), ia.idx.cuda(), ia.out.cuda()) if dev is None else dev
    out = out0.clone()
    dgr.det_index_add(out, src, idx, seg_tile=seg_tile, ws=ws, bad_count=bad)
    return out


CASES = [
    # N, D, R, seg_tile, init
    (20000, 128, 700, 128, "zeros"),
    (20000, 128, 700, 1, "zeros"),
    (5000, 32, 100, 2, "random"),
    (5000, 32, 100, 4, "random"),
    (5000, 16, 100, 8, "random"),
    (9000, 64, 40, 32, "random"),
    (9000, 64, 40, 64, "random"),
    (30000, 256, 3000, 128, "random"),   # two column blocks
    (3000, 8, 5000, 128, "random"),      # most rows empty
    (4000, 4, 0, 128, "zeros"),          # only the dummy row
    (1, 4, 3, 128, "random"),
    (70000, 128, 60000, 128, "zeros"),   # many high-byte buckets
    (9000, 64, 40, 128, "random"),       # rows of ~200: split, folded by one warp
    (100000, 32, 20, 128, "random"),     # rows of ~4500: split, 21 rows over 16 fold blocks
    (60000, 256, 30, 128, "random"),     # split rows over two column blocks
    (50000, 128, 1, 128, "zeros"),       # one long row and the dummy row
]


@pytest.mark.parametrize("N,D,R,W,init", CASES)
def test_parity_small(N, D, R, W, init):
    ia = gi.index_add_input(N, D, R, seed=500 + N + R + W, out_init=init)
    want, _ = _oracle(ia, W)
    assert_bits_equal(_gpu(ia, W).cpu().numpy(), want, f"index_add N={N} D={D} R={R} W={W}")


@pytest.mark.parametrize("W", [128, 1])
def test_heavy_rows_split_path(W):
    # a skewed index: two rows take thousands of members (split into tiles
    # across warps for W = 128), plus 30 % padding
    g = torch.Generator().manual_seed(77)
    N, D, R = 40000, 128, 500
    idx = torch.randint(0, R, (N,), generator=g, dtype=torch.int64)
    idx[torch.randperm(N, generator=g)[:8000]] = 3
    idx[torch.randperm(N, generator=g)[:3000]] = R - 1
    idx[torch.randperm(N, generator=g)[:12000]] = -1
    ia = gi.IndexAddInput(torch.randn((N, D), generator=g), idx.to(torch.int32),
                          torch.randn((R + 1, D), generator=g), R)
    want, _ = _oracle(ia, W)
    assert_bits_equal(_gpu(ia, W).cpu().numpy(), want, f"heavy rows W={W}")


def test_bad_indices_counted_and_routed():
    ia = gi.index_add_input(10000, 16, 300, seed=8, pad_frac=0.05)
    idx = ia.idx.clone()
    idx[[1, 50, 999, 5000]] = torch.tensor([300, -7, 1 << 30, -(1 << 30)], dtype=torch.int32)
    ib = gi.IndexAddInput(ia.src, idx, ia.out, ia.R)
    want, bad = _oracle(ib)
    assert bad == 4
    badc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ws = dgr.workspace(dgr.index_add_workspace_bytes(10000, 300, 16))
    for _ in range(2):  # the workspace is reused; the count is overwritten, not summed
        got = _gpu(ib, ws=ws, bad=badc)
        assert_bits_equal(got.cpu().numpy(), want, "bad indices")
        assert int(badc.item()) == 4


def test_strided_rows():
    ia = gi.index_add_input(6000, 64, 200, seed=9, out_init="random")
    want, _ = _oracle(ia)
    src_wide = torch.full((6000, 96), float("nan"), device="cuda")
    src_wide[:, :64] = ia.src.cuda()
    out_wide = torch.full((201, 72), float("nan"), device="cuda")
    out_wide[:, :64] = ia.out.cuda()
    dgr.det_index_add(out_wide[:, :64], src_wide[:, :64], ia.idx.cuda())
    assert_bits_equal(out_wide[:, :64].cpu().numpy(), want, "strided")
    assert torch.isnan(out_wide[:, 64:]).all()


def test_empty():
    out = torch.randn(11, 8, device="cuda")
    ref = out.clone()
    badc = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    dgr.det_index_add(out, torch.zeros((0, 8), device="cuda"), torch.zeros(0, dtype=torch.int32, device="cuda"),
                      bad_count=badc)
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32)) and int(badc.item()) == 0


def test_full_workload_and_nondeterministic_control():
    ia = gi.index_add_full()
    want, bad = _oracle(ia)
    assert bad == 0
    dev = (ia.src.cuda(), ia.idx.cuda(), ia.out.cuda())
    ws = dgr.workspace(dgr.index_add_workspace_bytes(262144, 16384, 128))
    got = assert_replays_identical(lambda: _gpu(ia, dev=dev, ws=ws), n=20)
    assert_bits_equal(got.view(np.float32), want, "index_add full")
    assert dgr.read_device_status(ws) == 0
    # the replay check is not vacuous here: torch's atomic index_add_ on the
    # same data changes bits between runs
    src, idx, out0 = dev
    key = torch.where(idx < 0, torch.full_like(idx, 16384), idx).long()
    patterns = set()
    for _ in range(8):
        o = out0.clone()
        o.index_add_(0, key, src)
        torch.cuda.synchronize()
        patterns.add(hash(o.view(torch.int32).cpu().numpy().tobytes()))
    assert len(patterns) > 1


def test_workspace_reused_with_fewer_columns():
    # a workspace zeroed once for (N, R, D) serves calls of the same N and R
    # with any D' <= D, in any order; a call with no columns still sorts and
    # counts, and must leave every counter cleared like any other call
    for i, (N, D, R) in enumerate([(70000, 128, 60000), (3000, 8, 5000), (20000, 64, 700)]):
        ws = dgr.workspace(dgr.index_add_workspace_bytes(N, R, D))
        badc = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        ia = gi.index_add_input(N, D, R, seed=900 + i, out_init="random")
        idx = ia.idx.clone()
        idx[[0, N // 2]] = torch.tensor([R + 5, -3], dtype=torch.int32)
        ib = gi.IndexAddInput(ia.src, idx, ia.out, R)
        want, bad = _oracle(ib)
        half = gi.IndexAddInput(ib.src[:, :D // 2].contiguous(), idx, ib.out[:, :D // 2].contiguous(), R)
        want_half, _ = _oracle(half)
        assert bad == 2
        src, idx_d = ib.src.cuda(), ib.idx.cuda()
        for rep in range(2):
            # no columns (through the C ABI: torch gives a zero-element view
            # a null pointer): only the bad-index count comes out
            wide = torch.zeros((R + 1, 4), device="cuda")
            rc = dgr.lib().dgr_det_index_add(wide.data_ptr(), R, 0, 4, src.data_ptr(), D, idx_d.data_ptr(), N, 128,
                                             badc.data_ptr(), ws.data_ptr(), ws.numel(), None)
            assert rc == 0
            assert int(badc.item()) == 2 and torch.count_nonzero(wide) == 0
            got = _gpu(ib, dev=(src, idx_d, ib.out.cuda()), ws=ws, bad=badc)
            assert_bits_equal(got.cpu().numpy(), want, f"N={N} D={D} R={R} after a no-column call")
            assert int(badc.item()) == 2
            got = _gpu(half, ws=ws)
            assert_bits_equal(got.cpu().numpy(), want_half, f"N={N} D={D // 2} R={R} in a D={D} workspace")
        assert dgr.read_device_status(ws) == 0


def test_workspace_of_other_sizes_is_refused():
    # a workspace records the N and R of its first call; a call with other
    # sizes would read the first call's sorted keys as its counters, so it is
    # refused on the device: DGR_ERR_INVALID_ARG in the status word, out and
    # the bad-index count untouched, the workspace itself unchanged
    big = gi.index_add_input(70000, 128, 60000, seed=950, out_init="zeros")
    small = gi.index_add_input(3000, 8, 5000, seed=951, out_init="random")
    ws = dgr.workspace(dgr.index_add_workspace_bytes(70000, 60000, 128))
    assert ws.numel() >= dgr.index_add_workspace_bytes(3000, 5000, 8)
    want_big, _ = _oracle(big)
    assert_bits_equal(_gpu(big, ws=ws).cpu().numpy(), want_big, "first call")
    assert dgr.read_device_status(ws) == 0
    snapshot = ws.clone()
    badc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    out0 = small.out.cuda()
    got = _gpu(small, dev=(small.src.cuda(), small.idx.cuda(), out0), ws=ws, bad=badc)
    assert dgr.read_device_status(ws) == 1  # DGR_ERR_INVALID_ARG
    assert torch.equal(got.view(torch.int32), out0.view(torch.int32))
    assert int(badc.item()) == -7
    assert torch.equal(ws[256:], snapshot[256:])  # past the header: nothing written
    # the status cleared, the workspace still serves its own sizes
    assert dgr.read_device_status(ws, clear=True) == 1
    assert_bits_equal(_gpu(big, ws=ws).cpu().numpy(), want_big, "first sizes again")
    assert dgr.read_device_status(ws) == 0
    # zeroed, it serves the other sizes
    ws.zero_()
    want_small, _ = _oracle(small)
    assert_bits_equal(_gpu(small, ws=ws).cpu().numpy(), want_small, "other sizes after zeroing")
    assert dgr.read_device_status(ws) == 0
