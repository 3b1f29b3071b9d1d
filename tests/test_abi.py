"""The C ABI: the library builds, loads and exports every entry point that
include/*.h declares, and rejects bad arguments on the host before it touches
the GPU (these calls never reach the device, so they run without one)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import deterministic_gradient_reduction_gb300 as dgr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(dgr_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    dgr.build()
    return dgr.lib()


def test_header_declares_every_operation():
    names = declared_functions()
    for op in ("dgr_ordered_colsum", "dgr_ordered_rowdot_dprob", "dgr_det_index_add",
               "dgr_grouped_wgrad_accumulate", "dgr_grouped_dbias", "dgr_topk_canonicalize", "dgr_aux_loss",
               "dgr_dsrelu_dprob", "dgr_ordered_colsum_noalloc", "dgr_colsum_noalloc_read_status",
               "dgr_tc_probe_k16", "dgr_diag_wait_timeout", "dgr_diag_noalloc_wait_timeout"):
        assert op in names


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", dgr._LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(L, n) is not None


def test_library_is_built_for_sm_103a_only():
    out = subprocess.run(["cuobjdump", "--list-elf", dgr._LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    archs = set(re.findall(r"sm_(\d+a?)", out.stdout))
    assert archs == {"103a"}, archs


def test_status_strings_and_version(L):
    assert L.dgr_version() >= 103
    for code, name in dgr.STATUS.items():
        assert L.dgr_status_string(code).decode() == name
    assert L.dgr_status_string(99).decode() == "DGR_ERR_UNKNOWN"


def test_status_reads_refuse_a_null_workspace(L):
    # checked before any CUDA call
    st = ctypes.c_int32(-1)
    assert L.dgr_read_device_status(None, 0, ctypes.byref(st), None) == 1  # DGR_ERR_INVALID_ARG
    assert L.dgr_query_device_status(None, None) == 1


def test_workspace_sizes(L):
    # colsum: header + ready counters + [tiles x H] fp32 slots
    assert dgr.colsum_workspace_bytes(8388608, 64) >= 65536 * 64 * 4
    assert dgr.colsum_workspace_bytes(2048, 16) >= 16 * 16 * 4
    assert dgr.colsum_workspace_bytes(0, 16) >= 256
    assert dgr.colsum_workspace_bytes(100, 16, 3) == 0  # not a power of two
    assert dgr.rowdot_workspace_bytes(65536, 4096) == 0
    n = dgr.index_add_workspace_bytes(262144, 16384, 128)
    assert n >= 4 * 262144 * 4 + (16384 + 2) * 4
    assert dgr.index_add_workspace_bytes(10, 70000, 4) == 0  # R + 1 beyond the limit
    assert dgr.wgrad_workspace_bytes(8, 4096, 2048) >= 256


def _p(v):
    return ctypes.c_void_p(v)


def test_host_rejects_bad_arguments_before_any_launch(L):
    fake = _p(0x10000)  # never dereferenced: every call below fails validation first
    out = _p(0x20000)
    # colsum: bad dtype, non power-of-two tile, negative size, H beyond the limit
    assert L.dgr_ordered_colsum(fake, 7, 1, 4, 4, 16, 4, out, 0, 128, fake, 1 << 20, None) == 1
    assert L.dgr_ordered_colsum(fake, 1, 1, 4, 4, 16, 4, out, 0, 100, fake, 1 << 20, None) == 1
    assert L.dgr_ordered_colsum(fake, 1, -1, 4, 4, 16, 4, out, 0, 128, fake, 1 << 20, None) == 1
    assert L.dgr_ordered_colsum(fake, 1, 1, 4, 5000, 5000, 5000, out, 0, 128, fake, 1 << 20, None) == 2
    # workspace too small, misaligned workspace
    assert L.dgr_ordered_colsum(fake, 1, 1, 4096, 16, 0, 16, out, 0, 128, fake, 16, None) == 3
    assert L.dgr_ordered_colsum(fake, 1, 1, 4096, 16, 0, 16, out, 0, 128, _p(0x30008), 1 << 20, None) == 5
    # out overlapping the input
    assert L.dgr_ordered_colsum(_p(0x20000), 1, 1, 64, 16, 0, 16, _p(0x20010), 0, 128, _p(0x900000),
                                1 << 20, None) == 4
    # rowdot: only tile 128, ld smaller than N, overlap of dprob and dY
    assert L.dgr_ordered_rowdot_dprob(fake, fake, 1, 4, 256, 256, 256, out, 0, 64, None, None, 0, None) == 1
    assert L.dgr_ordered_rowdot_dprob(fake, fake, 1, 4, 256, 100, 256, out, 0, 128, None, None, 0, None) == 1
    assert L.dgr_ordered_rowdot_dprob(_p(0x100000), _p(0x200000), 1, 4, 256, 256, 256, _p(0x100100), 0, 128,
                                      None, None, 0, None) == 4
    # index_add: seg_tile not a power of two, R too large, D not a multiple of 4
    assert L.dgr_det_index_add(out, 10, 8, 8, fake, 8, fake, 4, 3, None, fake, 1 << 20, None) == 1
    assert L.dgr_det_index_add(out, 70000, 8, 8, fake, 8, fake, 4, 128, None, fake, 1 << 20, None) == 2
    assert L.dgr_det_index_add(_p(0x40000), 10, 6, 6, _p(0x80000), 6, fake, 4, 128, None, fake, 1 << 20,
                               None) == 5
    # index_add: workspace too small
    assert L.dgr_det_index_add(_p(0x40000), 10, 8, 8, _p(0x80000), 8, _p(0xC0000), 4, 128, None, _p(0x100000),
                               64, None) == 3
    # dbias: bad dtype, tile not a power of two, E = 0, E beyond the limit, tile below 8
    dy, offs, db = _p(0x100000), _p(0x200000), _p(0x300000)
    ws = _p(0x400000)
    assert L.dgr_grouped_dbias(dy, 7, 256, 16, 16, offs, 2, db, 16, 0, 128, ws, 1 << 20, None) == 1
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 2, db, 16, 0, 100, ws, 1 << 20, None) == 1
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 0, db, 16, 0, 128, ws, 1 << 20, None) == 1
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 2000, db, 16, 0, 128, ws, 1 << 20, None) == 2
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 2, db, 16, 0, 4, ws, 1 << 20, None) == 2
    # dbias: H not a multiple of 8 bf16 elements, workspace too small, dbias overlapping dY
    assert L.dgr_grouped_dbias(dy, 1, 256, 12, 12, offs, 2, db, 12, 0, 128, ws, 1 << 20, None) == 5
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 2, db, 16, 0, 128, ws, 64, None) == 3
    assert L.dgr_grouped_dbias(dy, 1, 256, 16, 16, offs, 2, _p(0x100040), 16, 0, 128, ws, 1 << 20, None) == 4
    # wgrad: chunk other than 512, N not a multiple of 128, E * N beyond 32-bit rows of main_grad
    g, x, mg = _p(0x100000), _p(0x200000), _p(0x300000)
    assert L.dgr_grouped_wgrad_accumulate(g, x, offs, 2, 1024, 128, 256, mg, 256, ws, 1 << 20, None) == 1
    assert L.dgr_grouped_wgrad_accumulate(g, x, offs, 2, 1024, 100, 256, mg, 512, ws, 1 << 20, None) == 2
    assert L.dgr_grouped_wgrad_accumulate(g, x, offs, 4096, 1024, 1 << 20, 256, mg, 512, ws, 1 << 20, None) == 2


def test_dbias_workspace_size(L):
    # header + FP32 partials [ceil(T / W) + E tiles, H]
    n = dgr.dbias_workspace_bytes(65536, 2048, 8)
    assert n >= 256 + (512 + 8) * 2048 * 4
    assert dgr.dbias_workspace_bytes(100, 16, 0) == 0
    assert dgr.dbias_workspace_bytes(100, 16, 2, 3) == 0


def test_topk_host_checks(L):
    a, b, c, d, e = (_p(x) for x in (0x100000, 0x200000, 0x300000, 0x400000, 0x500000))
    assert L.dgr_topk_canonicalize(a, 128, b, 128, 10, 0, c, d, e, 128, None) == 1     # K = 0
    assert L.dgr_topk_canonicalize(a, 300, b, 300, 10, 300, c, d, e, 300, None) == 2   # K beyond 256
    assert L.dgr_topk_canonicalize(a, 100, b, 128, 10, 128, c, d, e, 128, None) == 1   # ld below K
    assert L.dgr_topk_canonicalize(a, 128, b, 128, 10, 128, _p(0x100100), d, e, 128, None) == 4  # output on input
    assert L.dgr_topk_canonicalize(a, 128, b, 128, 10, 128, c, c, e, 128, None) == 4   # outputs overlap
    assert L.dgr_topk_canonicalize(_p(0x100002), 128, b, 128, 10, 128, c, d, e, 128, None) == 5


def test_aux_loss_host_checks(L):
    pr, tp, o, ws = _p(0x100000), _p(0x200000), _p(0x300000), _p(0x400000)
    F = ctypes.c_float
    assert L.dgr_aux_loss(pr, 10, 0, 8, tp, F(1.0), o, ws, 1 << 20, None) == 1       # E = 0
    assert L.dgr_aux_loss(pr, 10, 2000, 2000, tp, F(1.0), o, ws, 1 << 20, None) == 2  # E beyond 1024
    assert L.dgr_aux_loss(pr, 10, 8, 4, tp, F(1.0), o, ws, 1 << 20, None) == 1       # ld below E
    assert L.dgr_aux_loss(pr, 1000, 8, 8, tp, F(1.0), o, ws, 16, None) == 3          # workspace too small
    assert L.dgr_aux_loss(pr, 10, 8, 8, tp, F(1.0), _p(0x100004), ws, 1 << 20, None) == 4  # out inside probs
    assert dgr.aux_loss_workspace_bytes(65536) == 256 + 512 * 4


def test_dsrelu_host_checks(L):
    a, b, o, y, d, ws = (_p(x) for x in (0x1000000, 0x2000000, 0x3000000, 0x4000000, 0x5000000, 0x6000000))
    assert L.dgr_dsrelu_dprob(a, b, o, 0, 100, 64, 256, y, d, 0, ws, 1 << 30, None) == 1    # E = 0
    assert L.dgr_dsrelu_dprob(a, b, o, 2, 100, 60, 256, y, d, 0, ws, 1 << 30, None) == 2    # K not a multiple of 64
    assert L.dgr_dsrelu_dprob(a, b, o, 2, 100, 64, 300, y, d, 0, ws, 1 << 30, None) == 2    # N not a multiple of 256
    assert L.dgr_dsrelu_dprob(_p(0x1000008), b, o, 2, 100, 64, 256, y, d, 0, ws, 1 << 30, None) == 5  # A misaligned
    assert L.dgr_dsrelu_dprob(a, b, o, 2, 100, 64, 256, y, d, 0, ws, 64, None) == 3          # workspace too small
    assert L.dgr_dsrelu_dprob(a, b, o, 2, 100, 64, 256, y, _p(0x4000100), 0, ws, 1 << 30, None) == 4  # dprob in dY
    assert dgr.dsrelu_dprob_workspace_bytes(16384, 4096) == 256 + 16384 * 32 * 4


def test_wait_timeout_diag_host_checks(L):
    ws = _p(0x100000)
    assert L.dgr_diag_wait_timeout(2, 1000, ws, 256, None) == 1       # unknown wait
    assert L.dgr_diag_wait_timeout(0, 0, ws, 256, None) == 1          # no time at all
    assert L.dgr_diag_wait_timeout(0, 1000, ws, 64, None) == 3        # workspace below the header
    assert L.dgr_diag_wait_timeout(0, 1000, _p(0x100008), 256, None) == 5


def test_noalloc_host_checks(L):
    # the no-alloc column sum checks every argument before it touches its
    # static scratch (no device is needed to see these refusals)
    fake, out = _p(0x10000), _p(0x20000)
    assert L.dgr_ordered_colsum_noalloc(fake, 7, 1, 4, 4, 16, 4, out, 0, 128, None) == 1        # bad dtype
    assert L.dgr_ordered_colsum_noalloc(fake, 1, 1, 4, 4, 16, 4, None, 0, 128, None) == 1       # null out
    assert L.dgr_ordered_colsum_noalloc(fake, 1, 1, 4, 4, 16, 4, out, 0, 100, None) == 1        # tile not pow2
    assert L.dgr_ordered_colsum_noalloc(fake, 1, 1, 1 << 20, 512, 512 * (1 << 20), 512, out, 0, 128,
                                        None) == 3                                               # beyond scratch
    assert L.dgr_ordered_colsum_noalloc(_p(0x20000), 1, 1, 64, 16, 0, 16, _p(0x20010), 0, 128, None) == 4
    assert L.dgr_ordered_colsum_noalloc(_p(0x10001), 1, 1, 64, 16, 0, 16, out, 0, 128, None) == 5  # x misaligned
    assert L.dgr_colsum_noalloc_read_status(0, None, None) == 1
    assert L.dgr_diag_noalloc_wait_timeout(2, 1000, None) == 1


def test_colsum_launch_plan(L):
    # the column sum's folders wait for its producers, so one launch holds
    # both only when all folders and a producer can be resident at once;
    # otherwise producers and folders run as two launches
    plan = (ctypes.c_int32 * 4)()

    def p(T, H, W=128, dtype=1, vec=1, sms=152, occ=4, cap=0):
        assert L.dgr_diag_colsum_plan(T, H, W, dtype, vec, sms, occ, cap, plan) == 0
        return tuple(plan)

    # at most 512 tiles: one launch of 4-warp CTAs, the last warp folds
    assert p(2048, 16) == (0, 1, 4, 0)
    assert p(8192, 64) == (0, 1, 16, 0)
    assert p(8192, 64, cap=3) == (0, 1, 3, 0)
    assert p(65536, 64) == (0, 1, 128, 0)
    assert p(65536, 64, cap=5) == (0, 1, 5, 0)
    # 65536 tiles of 64 bf16 columns: 16 folders and 136 persistent producers
    assert p(8388608, 64) == (1, 1, 136, 16)
    assert p(8388608, 64, sms=17) == (1, 1, 1, 16)       # just enough SMs
    assert p(8388608, 64, sms=16) == (1, 2, 16, 16)      # a green context of 16 SMs: two launches
    assert p(8388608, 64, cap=8) == (1, 2, 8, 8)         # the diagnostic grid cap
    assert p(8388608, 64, cap=1) == (1, 2, 1, 1)
    # H = 520: CTA producers, 44 folders
    path, launches, prod, fold = p(70000, 520)
    assert (path, launches, fold) == (2, 1, 44) and prod > 0
    assert p(70000, 520, sms=8, occ=4)[:2] == (2, 2)     # 32 CTA slots < 45
    assert p(70000, 520, cap=44)[1] == 2
    assert p(0, 64) == (-1, 0, 0, 0)
    assert L.dgr_diag_colsum_plan(100, 0, 128, 1, 1, 152, 1, 0, plan) == 1
    assert L.dgr_diag_set_schedule(3, 0, 0) == 1 and L.dgr_diag_set_schedule(0, 0, -1) == 1


def test_diagnostic_entries_check_their_arguments(L):
    # refused before any device work: role, stall count and limit out of range,
    # and the packed-arithmetic pin's pointers
    f = _p(0x100000)
    for role, after, limit in ((0, 1, 100), (4, 1, 100), (1, -1, 100), (1, 1, 0), (1, 1, 2000000)):
        assert L.dgr_diag_wgrad_stall(f, f, f, 2, 1024, 128, 256, f, f, 1 << 20, role, after, limit, None) == 1
        assert L.dgr_diag_dsrelu_stall(f, f, f, 2, 1024, 64, 256, f, f, f, 1 << 20, role, after, limit, None) == 1
    assert L.dgr_diag_packed_ops(None, f, 4, f, f, None) == 1           # a null operand
    assert L.dgr_diag_packed_ops(f, f, -1, f, f, None) == 1             # a negative count
    assert L.dgr_diag_packed_ops(_p(0x100004), f, 4, f, f, None) == 5  # not 8-byte aligned
