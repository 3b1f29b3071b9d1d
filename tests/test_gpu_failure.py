"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every device-side wait of the library (the integer-counter waits of the
column-sum folders and the index_add fold blocks, the mbarrier waits of the
tensor-core pipelines) gives up after a time limit, records DGR_ERR_TIMEOUT in
the workspace status word and returns. Here each kind is made to run out on
purpose (it waits for something that nothing completes, with a limit of
milliseconds instead of the path's 2 s): the call returns, the host reads the
status and where it gave up, and the same context then runs a reduction
bit-exactly.
"""
import time

import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from util import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])
def test_wait_runs_out_and_the_context_stays_usable(which):
    ws = dgr.workspace(256)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = dgr.lib().dgr_diag_wait_timeout(which, 20000, ws.data_ptr(), ws.numel(), None)
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert 0.015 <= elapsed < 2.0  # it waited about its 20 ms, and no longer than the path's limit
    assert dgr.read_device_status(ws) == 7  # DGR_ERR_TIMEOUT
    assert dgr.query_device_status(ws) == 7  # the same word as a return value, left as it is
    where = int(ws[4:8].view(torch.int32).item())
    assert where == 90 + which
    assert dgr.read_device_status(ws, clear=True) == 7 and dgr.read_device_status(ws) == 0
    assert dgr.query_device_status(ws) == 0
    # the context is still usable: a column sum, bit-exact
    ci = gi.colsum_input(1, 3000, 64, seed=5)
    want = np.zeros(64, np.float32)
    oracle.ordered_colsum(gi.bits(ci.base), 1, 3000, 64, ci.stride_b, ci.stride_s, want)
    out = torch.zeros(64, device="cuda")
    dgr.ordered_colsum(ci.base.cuda().view(1, 3000, 64), out)
    assert_bits_equal(out.cpu().numpy(), want, "colsum after a timeout")


@pytest.mark.parametrize("role,after", [(1, 9), (1, 25), (2, 0), (2, 9), (2, 25), (3, 0), (3, 1)])
def test_wgrad_pipeline_role_times_out_and_drains(role, after):
    # one role of the tensor-core pipeline (1 TMA producer, 2 MMA issuer, 3 an
    # epilogue warp) of CTA 0 waits on a barrier nobody arrives at, mid-run
    # (256 tiles: CTA 0 takes two, of 18 and 15 stages): the call returns, the status
    # names the role, and the CTA's drains (copies in flight, issued MMAs,
    # reduce-adds) let it free TMEM and exit; the context then runs the wgrad
    # bit-exactly
    counts = [1100, 900]
    N, K = 2048, 2048
    wi = gi.wgrad_input(2, sum(counts), N, K, seed=41, dist="ternary", counts=counts)
    G, X, offs, mg = wi.G.cuda(), wi.X.cuda(), wi.offs.cuda(), wi.main_grad.cuda()
    ws = dgr.workspace(256)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = dgr.lib().dgr_diag_wgrad_stall(G.data_ptr(), X.data_ptr(), offs.data_ptr(), 2, sum(counts), N, K,
                                         mg.data_ptr(), ws.data_ptr(), ws.numel(), role, after, 20000, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 2.0
    assert dgr.read_device_status(ws) == 7  # DGR_ERR_TIMEOUT
    assert int(ws[4:8].view(torch.int32).item()) == 14 + role
    out = wi.main_grad.cuda()
    dgr.grouped_wgrad_accumulate(G, X, offs, out)
    Gd, Xd = wi.G.to(torch.float64).numpy(), wi.X.to(torch.float64).numpy()
    want = wi.main_grad.to(torch.float64).numpy().copy()
    o = wi.offs.numpy()
    for e in range(2):
        want[e] += Gd[o[e]:o[e + 1]].T @ Xd[o[e]:o[e + 1]]
    assert_bits_equal(out.cpu().numpy(), want.astype(np.float32), "wgrad after a pipeline timeout")


def test_wgrad_stall_count_never_reached_changes_nothing():
    # a stall point past the end of the run: an ordinary call, status clear
    counts = [700, 300]
    wi = gi.wgrad_input(2, sum(counts), 128, 256, seed=42, dist="ternary", counts=counts)
    G, X, offs, mg = wi.G.cuda(), wi.X.cuda(), wi.offs.cuda(), wi.main_grad.cuda()
    ws = dgr.workspace(256)
    rc = dgr.lib().dgr_diag_wgrad_stall(G.data_ptr(), X.data_ptr(), offs.data_ptr(), 2, sum(counts), 128, 256,
                                         mg.data_ptr(), ws.data_ptr(), ws.numel(), 2, 1 << 30, 20000, None)
    assert rc == 0
    assert dgr.read_device_status(ws) == 0
    ref = wi.main_grad.cuda()
    dgr.grouped_wgrad_accumulate(G, X, offs, ref)
    assert torch.equal(mg.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("role,after", [(1, 5), (1, 12), (2, 0), (2, 5), (2, 12), (3, 0), (3, 1)])
def test_dsrelu_pipeline_role_times_out_and_drains(role, after):
    # the fused dsReLU dprob GEMM's roles, as for wgrad: 272 tiles, so CTA 0
    # takes two of 8 stages each; the call returns, the status names the role,
    # the CTA drains and exits, and the context then computes dprob bit-exactly
    counts = [1100, 900]
    T, K, N = sum(counts), 512, 4096
    ds = gi.dsrelu_input(2, T, K, N, seed=43, counts=counts)
    A, B, offs, dY = ds.A.cuda(), ds.B.cuda(), ds.offs.cuda(), ds.dY.cuda()
    dp = torch.zeros(T, device="cuda")
    ws = dgr.workspace(dgr.dsrelu_dprob_workspace_bytes(T, N))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = dgr.lib().dgr_diag_dsrelu_stall(A.data_ptr(), B.data_ptr(), offs.data_ptr(), 2, T, K, N, dY.data_ptr(),
                                          dp.data_ptr(), ws.data_ptr(), ws.numel(), role, after, 20000, None)
    assert rc == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 2.0
    assert dgr.read_device_status(ws) == 7  # DGR_ERR_TIMEOUT
    assert int(ws[4:8].view(torch.int32).item()) == 40 + role
    # the context still works: the smoke's case against the oracle, bit for bit
    sm = gi.dsrelu_input(2, 128, 64, 256, seed=9, counts=[100, 28])
    want = np.zeros(128, np.float32)
    oracle.dsrelu_dprob(gi.bits(sm.A), gi.bits(sm.B), sm.offs.numpy(), gi.bits(sm.dY), want)
    got = torch.zeros(128, device="cuda")
    dgr.dsrelu_dprob(sm.A.cuda(), sm.B.cuda(), sm.offs.cuda(), sm.dY.cuda(), got)
    assert_bits_equal(got.cpu().numpy(), want, "dsrelu dprob after a pipeline timeout")
