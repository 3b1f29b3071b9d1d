"""No output bit depends on how the work is handed out on the GPU.

The pages' determinism bug (cuDNN-frontend PR #521, commit "deterministic
dprob") was an accumulation whose order followed the schedule: a loop whose
direction depended on the pipeline phase, and atomics across CTAs. Here every
operation is run again with its work items (tiles, rows, warp shares) handed
out in descending and in seeded shuffled order, with the grid capped (down to
one CTA, where the column sum takes its two-launch form and index_add's long
rows are folded by warps), and on another stream; every output must keep the
default launch's bits, and the default launch's bits equal the CPU oracle's.
"""
import contextlib

import numpy as np
import pytest
import torch

import deterministic_gradient_reduction_gb300 as dgr
import dgr_inputs as gi
import oracle
from util import assert_bits_equal

pytestmark = pytest.mark.gpu

# (order, seed, grid cap): descending; shuffled; capped; shuffled and capped
# below the column sum's folder count (two launches); one CTA, descending
SCHEDULES = [(1, 0, 0), (2, 2024, 0), (0, 0, 37), (2, 99, 3), (1, 0, 1)]


@contextlib.contextmanager
def schedule(order, seed, cap):
    L = dgr.lib()
    assert L.dgr_diag_set_schedule(order, seed, cap) == 0
    try:
        yield
    finally:
        assert L.dgr_diag_set_schedule(0, 0, 0) == 0


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int32).cpu().numpy()


def check_every_schedule(run, what: str) -> np.ndarray:
    """run() enqueues one call on the current stream and returns its output;
    every schedule and a second stream must give the default launch's bits."""
    base = _bits(run())
    for sch in SCHEDULES:
        with schedule(*sch):
            got = _bits(run())
        diff = np.flatnonzero(got.reshape(-1) != base.reshape(-1))
        assert diff.size == 0, f"{what}: schedule {sch} changed {diff.size} outputs"
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        out = run()
    torch.cuda.current_stream().wait_stream(side)
    assert np.array_equal(_bits(out), base), f"{what}: another stream changed bits"
    return base


def _colsum_oracle(ci: gi.ColsumInput):
    out = np.zeros(ci.H, np.float32)
    flat = gi.bits(ci.base) if ci.base.dtype == torch.bfloat16 else gi.f32(ci.base)
    oracle.ordered_colsum(flat, ci.B, ci.S, ci.H, ci.stride_b, ci.stride_s, out)
    return out


@pytest.mark.parametrize("which", ["large", "small", "strided", "cta_path"])
def test_colsum(which):
    ci = {"large": gi.colsum_large, "small": gi.colsum_small, "strided": gi.colsum_strided,
          "cta_path": lambda: gi.colsum_input(1, 70000, 520, seed=61)}[which]()
    base = ci.base.cuda()
    x = base.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))

    def run():
        out = torch.zeros(ci.H, device="cuda")
        return dgr.ordered_colsum(x, out)

    got = check_every_schedule(run, f"colsum {which}")
    assert_bits_equal(got.view(np.float32), _colsum_oracle(ci), f"colsum {which} vs oracle")


def test_dprob():
    dp = gi.dprob_full()
    dY, Y = dp.dY.cuda(), dp.Y.cuda()

    def run():
        out = torch.zeros(dp.M, device="cuda")
        return dgr.ordered_rowdot_dprob(dY, Y, out)

    got = check_every_schedule(run, "dprob 65536x4096")
    want = np.zeros(dp.M, np.float32)
    oracle.ordered_rowdot_dprob(gi.bits(dp.dY).reshape(-1), gi.bits(dp.Y).reshape(-1), dp.M, dp.N, dp.N, dp.N, want)
    assert_bits_equal(got.view(np.float32), want, "dprob vs oracle")


def _index_add_oracle(ia: gi.IndexAddInput):
    out = gi.f32(ia.out).copy()
    N, D = ia.src.shape
    oracle.det_index_add(out, ia.R, D, D, gi.f32(ia.src), D, ia.idx.numpy(), N)
    return out


@pytest.mark.parametrize("which", ["full", "long_rows"])
def test_index_add(which):
    if which == "full":
        ia = gi.index_add_full()
    else:  # rows of thousands of members: split by tile, folded by fold blocks (or by warps on one CTA)
        ia = gi.index_add_input(100000, 32, 20, seed=620, out_init="random")
    src, idx, out0 = ia.src.cuda(), ia.idx.cuda(), ia.out.cuda()

    def run():
        out = out0.clone()
        return dgr.det_index_add(out, src, idx)

    got = check_every_schedule(run, f"index_add {which}")
    assert_bits_equal(got.view(np.float32), _index_add_oracle(ia), f"index_add {which} vs oracle")


def test_wgrad_full_workload():
    wi = gi.wgrad_full()
    G, X, offs, mg = wi.G.cuda(), wi.X.cuda(), wi.offs.cuda(), wi.main_grad.cuda()

    def run():
        out = mg.clone()
        return dgr.grouped_wgrad_accumulate(G, X, offs, out)

    check_every_schedule(run, "wgrad E8 T32768 N4096 K2048")


def test_wgrad_full_output_vs_oracle():
    counts = [700, 0, 1029, 300, 64]
    wi = gi.wgrad_input(len(counts), sum(counts), 256, 512, seed=1063, counts=counts)
    G, X, offs, mg = wi.G.cuda(), wi.X.cuda(), wi.offs.cuda(), wi.main_grad.cuda()

    def run():
        out = mg.clone()
        return dgr.grouped_wgrad_accumulate(G, X, offs, out)

    got = check_every_schedule(run, "wgrad small")
    want = gi.f32(wi.main_grad).copy()
    oracle.grouped_wgrad_accumulate(gi.bits(wi.G), gi.bits(wi.X), wi.offs.numpy(), wi.E, 256, 512, want)
    assert_bits_equal(got.view(np.float32), want, "wgrad small vs oracle")


def test_aux_loss():
    a = gi.aux_full()
    probs, tpe = a.probs.cuda(), a.tpe.cuda()
    got = check_every_schedule(lambda: dgr.aux_loss(probs, tpe, a.scale), "aux loss 65536x128")
    want = oracle.aux_loss(a.probs.numpy(), a.tpe.numpy(), a.scale)
    assert got.view(np.float32)[0].view(np.uint32) == want.view(np.uint32)


def test_dsrelu_dprob():
    counts = [300, 0, 213, 129]
    d = gi.dsrelu_input(len(counts), sum(counts), 128, 512, seed=1091, counts=counts)
    A, B, offs, dY = d.A.cuda(), d.B.cuda(), d.offs.cuda(), d.dY.cuda()

    def run():
        out = torch.zeros(sum(counts), device="cuda")
        return dgr.dsrelu_dprob(A, B, offs, dY, out)

    got = check_every_schedule(run, "dsrelu dprob")
    want = d.dprob.numpy().copy()
    oracle.dsrelu_dprob(gi.bits(d.A), gi.bits(d.B), d.offs.numpy(), gi.bits(d.dY), want)
    assert_bits_equal(got.view(np.float32), want, "dsrelu dprob vs oracle")
