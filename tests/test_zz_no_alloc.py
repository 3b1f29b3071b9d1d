"""The column sum for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: a plugin that only
receives input and output pointers from a host framework owning all device
memory, code running inside another allocator, or a hot path where a
cudaMalloc would stall the device. dgr_ordered_colsum_noalloc serves them
from a static scratch array inside the library. These tests call it through
the C ABI and require its output to equal the workspace form's bit for bit
(the tolerance every parity test here uses), on consecutive calls that share
the array, and require calls that need more scratch than the array holds to
be refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi

pytestmark = pytest.mark.gpu

P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
SCRATCH_BYTES = 4 << 20


def _noalloc():
    dgr.build()
    f = dgr.lib().dgr_ordered_colsum_noalloc
    f.argtypes = [P, I32, I64, I64, I64, I64, I64, P, I32, I32, P]
    f.restype = I32
    return f


def _call(f, x: torch.Tensor, out: torch.Tensor, accumulate=False, tile_rows=128) -> int:
    B, S, H = x.shape
    dt = dgr.DTYPE_BF16 if x.dtype == torch.bfloat16 else dgr.DTYPE_F32
    return f(x.data_ptr(), dt, B, S, H, x.stride(0), x.stride(1), out.data_ptr(), int(accumulate), tile_rows,
             torch.cuda.current_stream().cuda_stream)


def _input(B, S, H, seed, ts=None):
    ci = gi.colsum_input(B, S, H, seed=seed, token_stride=ts)
    base = ci.base.cuda()
    return base.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))


def _reference(x, out0=None, accumulate=False, tile_rows=128):
    out = torch.zeros(x.shape[2], device="cuda") if out0 is None else out0.clone()
    dgr.ordered_colsum(x, out, accumulate=accumulate, tile_rows=tile_rows)
    return out


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_matches_workspace_form_on_consecutive_calls():
    f = _noalloc()
    xa = _input(1, 2048, 16, seed=1)
    xb = _input(4, 2048, 64, seed=4, ts=128)
    for x in (xa, xb, xa):  # three calls in a row share the one scratch array
        out = torch.full((x.shape[2],), float("nan"), device="cuda")
        assert _call(f, x, out) == 0
        torch.cuda.synchronize()
        assert _same(out, _reference(x))
    out0 = torch.randn(64, device="cuda")
    for _ in range(2):
        out = out0.clone()
        assert _call(f, xb, out, accumulate=True, tile_rows=64) == 0
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
