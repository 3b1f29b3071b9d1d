"""The column sum for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: a plugin that only
receives input and output pointers from a host framework owning all device
memory, code running inside another allocator, or a hot path where a
cudaMalloc would stall the device. dgr_ordered_colsum_noalloc serves them
from a static scratch array inside the library. These tests call it through
the C ABI and require its output to equal, bit for bit, both the CPU oracle
and the workspace form, on consecutive calls that share the array; calls that
need more scratch than the array holds, or that have a bad argument, must be
refused before anything is enqueued; and a device-side error recorded in the
array must be visible through dgr_colsum_noalloc_read_status.
"""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from util import assert_bits_equal

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20


def _noalloc():
    dgr.build()
    return dgr.lib().dgr_ordered_colsum_noalloc


def _call(f, x: torch.Tensor, out: torch.Tensor, accumulate=False, tile_rows=128, dtype=None) -> int:
    B, S, H = x.shape
    dt = (dgr.DTYPE_BF16 if x.dtype == torch.bfloat16 else dgr.DTYPE_F32) if dtype is None else dtype
    return f(x.data_ptr(), dt, B, S, H, x.stride(0), x.stride(1), None if out is None else out.data_ptr(),
             int(accumulate), tile_rows, torch.cuda.current_stream().cuda_stream)


def _status(clear=False) -> int:
    st = ctypes.c_int32(-1)
    rc = dgr.lib().dgr_colsum_noalloc_read_status(int(clear), ctypes.byref(st),
                                                  torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    return st.value


def _input(B, S, H, seed, ts=None):
    ci = gi.colsum_input(B, S, H, seed=seed, token_stride=ts)
    base = ci.base.cuda()
    return ci, base.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))


def _oracle(ci, out0=None, accumulate=False, tile_rows=128):
    out = np.zeros(ci.H, np.float32) if out0 is None else out0.copy()
    oracle.ordered_colsum(gi.bits(ci.base), ci.B, ci.S, ci.H, ci.stride_b, ci.stride_s, out,
                          accumulate=accumulate, tile_rows=tile_rows)
    return out


def _reference(x, out0=None, accumulate=False, tile_rows=128):
    out = torch.zeros(x.shape[2], device="cuda") if out0 is None else out0.clone()
    dgr.ordered_colsum(x, out, accumulate=accumulate, tile_rows=tile_rows)
    return out


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_matches_oracle_and_workspace_form_on_consecutive_calls():
    f = _noalloc()
    ca, xa = _input(1, 2048, 16, seed=1)
    cb, xb = _input(4, 2048, 64, seed=4, ts=128)
    for ci, x in ((ca, xa), (cb, xb), (ca, xa)):  # three calls in a row share the one scratch array
        out = torch.full((x.shape[2],), float("nan"), device="cuda")
        assert _call(f, x, out) == 0
        assert _status() == 0
        assert_bits_equal(out.cpu().numpy(), _oracle(ci), "no-alloc colsum vs oracle")
        assert _same(out, _reference(x))
    out0 = torch.randn(64, device="cuda")
    for _ in range(2):
        out = out0.clone()
        assert _call(f, xb, out, accumulate=True, tile_rows=64) == 0
        assert_bits_equal(out.cpu().numpy(), _oracle(cb, out0.cpu().numpy(), True, 64), "accumulate vs oracle")
        assert _same(out, _reference(xb, out0, accumulate=True, tile_rows=64))


def test_refuses_calls_beyond_the_static_scratch():
    f = _noalloc()
    T, H = 1 << 20, 512  # needs about 16 MiB of slots
    assert dgr.colsum_workspace_bytes(T, H) > SCRATCH_BYTES
    x = torch.zeros((1, T, H), dtype=torch.bfloat16, device="cuda")
    out = torch.full((H,), 7.0, device="cuda")
    assert _call(f, x, out) == 3  # DGR_ERR_WORKSPACE_TOO_SMALL, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert _call(f, x[:, :1024], out) == 0  # a small call afterwards still works
    assert _same(out, _reference(x[:, :1024]))


def test_device_error_is_visible_and_refused_calls_touch_nothing():
    f = _noalloc()
    ci, x = _input(1, 2048, 16, seed=1)
    # a bounded wait on the array's status word runs out (20 ms), as a
    # column-sum folder's would: the caller sees DGR_ERR_TIMEOUT
    assert dgr.lib().dgr_diag_noalloc_wait_timeout(0, 20000, torch.cuda.current_stream().cuda_stream) == 0
    assert _status() == 7
    # refused calls enqueue nothing: the recorded status stays as it was
    out = torch.full((16,), 3.0, device="cuda")
    assert _call(f, x, out, dtype=7) == 1      # bad dtype
    assert _call(f, x, None) == 1              # null out
    assert _call(f, x, out, tile_rows=3) == 1  # tile not a power of two
    assert _status() == 7
    assert torch.all(out == 3.0)
    # the read can clear the word; the next call zeroes its region anyway
    assert _status(clear=True) == 7 and _status() == 0
    assert dgr.lib().dgr_diag_noalloc_wait_timeout(1, 20000, torch.cuda.current_stream().cuda_stream) == 0
    assert _status() == 7
    assert _call(f, x, out) == 0
    assert _status() == 0
    assert_bits_equal(out.cpu().numpy(), _oracle(ci), "after a recorded error")
