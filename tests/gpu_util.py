"""GPU test helpers: side-stream contention and bitwise replay checks."""
from __future__ import annotations

import contextlib

import numpy as np
import torch


@contextlib.contextmanager
def side_stream_contention(n_iter: int = 4):
    """Keep a second stream busy (bf16 matmuls and a 1 GiB copy) while the
    body enqueues its work on the current stream."""
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    src = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        for _ in range(n_iter):
            a = (a @ a).clamp_(-1, 1)
            dst.copy_(src)
    try:
        yield side
    finally:
        torch.cuda.synchronize()
        del a, src, dst


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int32).cpu().numpy()


def assert_replays_identical(run, n: int = 20, contention: bool = True) -> np.ndarray:
    """Run `run()` (returns an fp32 tensor) n times, half of them under side
    stream contention, and require every run's bit pattern to be identical."""
    first = None
    for i in range(n):
        ctx = side_stream_contention() if (contention and i % 2 == 1) else contextlib.nullcontext()
        with ctx:
            out = run()
        torch.cuda.synchronize()
        b = bits(out)
        if first is None:
            first = b
        else:
            diff = np.flatnonzero(b.reshape(-1) != first.reshape(-1))
            assert diff.size == 0, f"replay {i}: {diff.size} outputs changed bits"
    return first
