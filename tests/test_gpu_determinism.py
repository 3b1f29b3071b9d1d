"""Evidence that the replay tests could fail, and the side-stream regression.

Anti-vacuity (cuDNN-frontend PR #521, determinism-test review: the atomic
dprob was already bit-stable at small sizes, so a passing replay test there
proved nothing): at the full 1 GiB column sum and the 65536 x 4096 dprob, the
atomic reductions the pages replace (dgr_diag_atomic_colsum / _rowdot) must
change bits between runs on the same data, while the ordered ones do not.

Side stream (cuDNN-frontend PR #521, "Order the dprob reduction against the
kernel's stream"): a call made on a stream other than torch's current one, with
torch's stream busy and a same-sized allocator block poisoned, must still give
the oracle's bits. The test passes the stream explicitly and never enters
torch.cuda.stream(): inside it the two streams would be the same and a
misplaced step (a workspace zeroed on the wrong stream) could not show.
"""
import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from util import assert_bits_equal

pytestmark = pytest.mark.gpu


def _patterns(run, n=8) -> set:
    seen = set()
    for _ in range(n):
        out = run()
        torch.cuda.synchronize()
        seen.add(out.view(torch.int32).cpu().numpy().tobytes())
    return seen


def test_atomic_colsum_changes_bits_where_the_ordered_one_does_not():
    ci = gi.colsum_large()
    x = ci.base.cuda()
    T, H = ci.S, ci.H
    out_a = torch.empty(H, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def atomic():
        assert dgr.lib().dgr_diag_atomic_colsum(x.data_ptr(), T, H, out_a.data_ptr(), stream) == 0
        return out_a

    seen = _patterns(atomic)
    assert len(seen) > 1, "the atomic column sum gave one bit pattern in 8 runs"
    ws = dgr.workspace(dgr.colsum_workspace_bytes(T, H))
    out = torch.empty(H, device="cuda")
    assert len(_patterns(lambda: dgr.ordered_colsum(x.view(1, T, H), out, ws=ws))) == 1
    # the control computes the same sum, up to the order of its additions
    np.testing.assert_allclose(out_a.cpu().numpy(), out.cpu().numpy(), rtol=1e-4, atol=1e-3)


def test_atomic_dprob_changes_bits_where_the_ordered_one_does_not():
    dp = gi.dprob_full()
    dY, Y = dp.dY.cuda(), dp.Y.cuda()
    out_a = torch.empty(dp.M, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def atomic():
        assert dgr.lib().dgr_diag_atomic_rowdot(dY.data_ptr(), Y.data_ptr(), dp.M, dp.N, out_a.data_ptr(),
                                                stream) == 0
        return out_a

    seen = _patterns(atomic)
    assert len(seen) > 1, "the atomic dprob gave one bit pattern in 8 runs"
    out = torch.empty(dp.M, device="cuda")
    assert len(_patterns(lambda: dgr.ordered_rowdot_dprob(dY, Y, out))) == 1
    np.testing.assert_allclose(out_a.cpu().numpy(), out.cpu().numpy(), rtol=1e-4, atol=1e-2)


def _occupy_current_stream():
    """Tens of milliseconds of matmuls on torch's current stream."""
    a = torch.randn(8192, 8192, device="cuda", dtype=torch.bfloat16)
    for _ in range(40):
        a = (a @ a).clamp_(-1, 1)
    return a


def _poison(nbytes: int):
    """A block of the workspace's size, filled with 0xAB and freed on torch's
    current stream: a workspace wrongly taken from that stream's pool would be
    this block, zeroed only after the busy stream gets there."""
    p = torch.full((max(int(nbytes), 256),), 0xAB, dtype=torch.uint8, device="cuda")
    del p


def test_call_on_a_side_stream_with_torch_stream_busy_and_poisoned_block():
    side = torch.cuda.Stream()
    cases = []  # (name, workspace bytes, expected bits, call(output) on the side stream, initial output)
    # colsum: the ticket path and the folder path
    for ci in (gi.colsum_small(), gi.colsum_input(1, 200000, 64, seed=71)):
        base = ci.base.cuda()
        x = base.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))
        want = np.zeros(ci.H, np.float32)
        oracle.ordered_colsum(gi.bits(ci.base), ci.B, ci.S, ci.H, ci.stride_b, ci.stride_s, want)
        cases.append((f"colsum {ci.B}x{ci.S}x{ci.H}", dgr.colsum_workspace_bytes(ci.B * ci.S, ci.H), want,
                      lambda out, x=x: dgr.ordered_colsum(x, out, stream=side), torch.zeros(ci.H, device="cuda")))
    # index_add
    ia = gi.index_add_input(20000, 128, 700, seed=72, out_init="random")
    src, idx = ia.src.cuda(), ia.idx.cuda()
    want = gi.f32(ia.out).copy()
    oracle.det_index_add(want, ia.R, 128, 128, gi.f32(ia.src), 128, ia.idx.numpy(), 20000)
    cases.append(("index_add", dgr.index_add_workspace_bytes(20000, 700, 128), want,
                  lambda out: dgr.det_index_add(out, src, idx, stream=side), ia.out.cuda()))
    # aux loss (its output, too, is allocated by the binding, on the call's stream)
    a = gi.aux_input(5000, 128, seed=73)
    probs, tpe = a.probs.cuda(), a.tpe.cuda()
    want = np.array([oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), a.scale)], np.float32)
    cases.append(("aux_loss", dgr.aux_loss_workspace_bytes(5000), want,
                  lambda out: dgr.aux_loss(probs, tpe, a.scale, stream=side), None))
    for name, ws_bytes, want, call, out in cases:
        torch.cuda.synchronize()  # inputs and initial outputs are in place on every stream
        _poison(ws_bytes)
        busy = _occupy_current_stream()
        res = call(out)  # the binding allocates the workspace; nothing here enters torch.cuda.stream()
        side.synchronize()
        got = res.cpu().numpy()  # final: the side stream is done and nothing else writes it
        assert_bits_equal(got, want, f"{name} on a side stream")
        torch.cuda.synchronize()
        del busy

