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
