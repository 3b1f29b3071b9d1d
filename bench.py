#!/usr/bin/env python3
"""Benchmark of one deterministic-reduction step on GB300.

A step is one pass of every operation on its seeded synthetic workload, with
the inputs resident in HBM:
  colsum_large    ordered column sum, bf16 [8388608, 64] (1 GiB)  -> fp32 [64]
  colsum_small    ordered column sum, bf16 [2048, 16]             -> fp32 [16]
  dprob           ordered dprob, bf16 [65536, 4096] x 2 (1 GiB)   -> fp32 [65536]
  colsum_strided  ordered column sum, bf16 [4, 2048, 64] at token stride 128
  index_add       deterministic index_add, fp32 [262144, 128] -> [16385, 128]
  wgrad           grouped wgrad, E 8, T 32768, N 4096, K 2048, into fp32 main_grad
The order interleaves the small operations with large streams, and every step
moves several GB, far more than the 129 MB L2, so no operation finds its
inputs in L2 from the previous step (no separate flush is needed).

Printed (rank 0, one JSON line): the ordered-reduction throughput in GB/s
(algorithmic bytes of the five reductions over their device time, the five
run back to back K times between one pair of CUDA events), the wgrad
TFLOP/s, per-operation figures, the roofline of the dominant operation, the
end-to-end figure through host buffers, SM clocks sampled during the timed
region and the CPU oracle's own rate on the host cores.

`--impl reference` times the CPU oracle instead (the only reference this
project has): single-threaded C on the host cores, bounded samples per step.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dgr_inputs as gi  # noqa: E402

METRIC = "ordered-reduction HBM GB/s (% of peak), bitwise replay; wgrad TFLOP/s"
REDUCTIONS = ["colsum_large", "colsum_small", "dprob", "colsum_strided", "index_add"]

# algorithmic bytes (or flops) per call: inputs read once, outputs written once
ALGO = {
    "colsum_large": 8388608 * 64 * 2 + 64 * 4,
    "colsum_small": 2048 * 16 * 2 + 16 * 4,
    "dprob": 2 * 65536 * 4096 * 2 + 65536 * 4,
    "colsum_strided": 4 * 2048 * 64 * 2 + 64 * 4,
    "index_add": 262144 * 128 * 4 + 262144 * 4 + 2 * 16385 * 128 * 4,
    "wgrad_flop": 2 * 4096 * 2048 * 32768,
    "wgrad": 32768 * 4096 * 2 + 32768 * 2048 * 2 + 2 * 8 * 4096 * 2048 * 4,
    "dbias": 65536 * 2048 * 2 + 8 * 2048 * 4,
    "topk": 65536 * 128 * 4 * 5,
    "aux_loss": 65536 * 128 * 4 + 128 * 4 + 4,
    "dsrelu_flop": 2 * 16384 * 2048 * 4096,
}
LAUNCHES = {"colsum_large": 1, "colsum_small": 1, "dprob": 1, "colsum_strided": 1, "index_add": 4, "wgrad": 1,
            "dbias": 2, "topk": 1, "aux_loss": 1, "dsrelu": 2}
# operations beyond the step (the next rows of the scope), timed on their own after it
EXTRAS = ["dbias", "topk", "aux_loss", "dsrelu"]
# next rows whose inputs fit in L2 are timed over this many copies of their
# inputs, taken in turn, so that more than twice L2 (129 MB) streams between two
# uses of one copy
ROTATE = {"topk": 3, "aux_loss": 9}
L2_NEXT_ROWS = ("no flush: dbias and dsrelu inputs larger than L2; topk and aux_loss rotate over 3 and 9 "
                "copies of their inputs (> 2x L2 between two uses of one copy)")
EXTRA_WORKLOADS = {
    "dbias": "grouped dbias bf16 65536x2048, 8 experts (multinomial rows) -> fp32 [8, 2048]",
    "topk": "canonical compact top-K, 65536 rows x 128 slots (int32 ids, fp32 logits; 10 % padding)",
    "aux_loss": "router aux-loss scalar, fp32 probs 65536 x 128 with top-8 expert counts",
    "dsrelu": "dprob fused into the grouped dsReLU GEMM, bf16 A 16384x2048, B 8x2048x4096, dY 16384x4096",
}

WORKLOAD = ("deterministic reduction step: colsum bf16 8388608x64 + colsum bf16 2048x16 + dprob bf16 "
            "65536x4096 + colsum bf16 4x2048x64 (token stride 128) + index_add fp32 262144x128 -> 16385 rows "
            "+ grouped wgrad E8 T32768 N4096 K2048 into fp32 main_grad")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d.get("bf16_tflops_sustained"),
                "src": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "src": "fallback"}


def tensor_peak(peaks: dict, clocks: dict | None) -> tuple[float, str]:
    """The dense bf16 peak a tensor kernel's fraction is taken of: the burst figure when its timed
    window ran at full clock with no power cap (a short region), the sustained figure when the
    window shows the power cap or clocks held below maximum (a long, power-limited loop)."""
    c = clocks or {}
    sm, smax = c.get("sm_mhz"), c.get("sm_max_mhz")
    capped = "sw_power_cap" in (c.get("reasons") or []) or (sm is not None and smax and sm < 0.97 * smax)
    if capped and peaks.get("bf16_sus"):
        return peaks["bf16_sus"], "bf16 sustained"
    return peaks["bf16"], "bf16 burst"


# The sources each captured operation's kernels are built from: a capture's
# DRAM bytes hold only while these files are as they were when it was taken.
TRAFFIC_SOURCES = {
    "colsum_large": ["colsum.cu", "dgr_common.cuh"],
    "dprob": ["rowdot.cu", "dgr_common.cuh"],
    "index_add": ["index_add.cu", "dgr_common.cuh"],
    "wgrad": ["wgrad.cu", "tc_common.cuh", "dgr_common.cuh"],
    "dbias": ["dbias.cu", "dgr_common.cuh"],
    "topk": ["topk.cu", "dgr_common.cuh"],
    "aux_loss": ["aux_loss.cu", "dgr_common.cuh"],
}


def source_digest(op: str) -> str | None:
    """SHA-256 over the sources of op's kernels (TRAFFIC_SOURCES), or None."""
    import hashlib
    files = TRAFFIC_SOURCES.get(op)
    if not files:
        return None
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deterministic_gradient_reduction_gb300", "csrc")
    for f in files:
        path = os.path.join(csrc, f)
        if not os.path.isfile(path):
            return None
        h.update(f.encode() + b"\0" + open(path, "rb").read())
    return h.hexdigest()


def load_traffic() -> dict:
    """DRAM bytes per launch from the committed ncu summaries (profiles/*.md):
    a line `traffic: <op> <bytes>` per captured operation, kept only when the
    summary's `source: <op> <sha256>` line matches the kernels' sources as they
    are now (a figure taken on a kernel that has changed since is dropped)."""
    out = {}
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return out
    for f in sorted(os.listdir(d)):
        if f.endswith(".md"):
            text = open(os.path.join(d, f)).read()
            src = {m.group(1): m.group(2) for m in re.finditer(r"^source:\s*(\w+)\s+([0-9a-f]{64})\s*$", text, re.M)}
            for m in re.finditer(r"^traffic:\s*(\w+)\s+(\d+)\s*$", text, re.M):
                op = m.group(1)
                if src.get(op) is not None and src[op] == source_digest(op):
                    out[op] = int(m.group(2))
    return out


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        """End sampling; the clocks of the window between the two marks."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        return self.window(self.t0, self.t1, fallback=True)

    def window(self, t0, t1, fallback: bool = False) -> dict:
        """Median SM clock, maximum clock and throttle reasons of the samples taken in [t0, t1]
        (with `fallback`, of all samples when none falls inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [s for t, s in self.samples if t0 is None or (t0 <= t <= (t1 or t) + 0.15)]
        if not inside and fallback:
            inside = [s for _, s in self.samples]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def make_ops(dev, torch, dgr, with_wgrad, only=None, small=False):
    """Build device inputs and one closure per operation (enqueue only).
    `only` keeps one operation; `small` shrinks colsum_large, dprob and wgrad
    (fewer tokens / rows, same widths) for profiler captures."""
    ops, host, outs, rotations = {}, {}, {}, {}
    want = (lambda n: only is None or n == only)

    gens = {"colsum_large": (gi.colsum_large if not small else
                             (lambda: gi.colsum_input(1, 2097152, 64, seed=4, scale=0.02))),
            "colsum_small": gi.colsum_small, "colsum_strided": gi.colsum_strided}
    for name, gen in gens.items():
        if not want(name):
            continue
        ci = gen()
        base = ci.base.to(dev)
        x = base.as_strided((ci.B, ci.S, ci.H), (ci.stride_b, ci.stride_s, 1))
        out = torch.zeros(ci.H, device=dev)
        ws = dgr.workspace(dgr.colsum_workspace_bytes(ci.B * ci.S, ci.H), dev)
        ops[name] = (lambda x=x, out=out, ws=ws: dgr.ordered_colsum(x, out, ws=ws))
        host[name] = ([ci.base], [base])
        outs[name] = out
    if want("dprob"):
        dp = gi.dprob_full() if not small else gi.dprob_input(16384, 4096, seed=3)
        dY, Y = dp.dY.to(dev), dp.Y.to(dev)
        dprob = torch.zeros(dp.M, device=dev)
        ops["dprob"] = lambda dY=dY, Y=Y, dprob=dprob: dgr.ordered_rowdot_dprob(dY, Y, dprob)
        host["dprob"] = ([dp.dY, dp.Y], [dY, Y])
        outs["dprob"] = dprob
    if want("index_add"):
        ia = gi.index_add_full()
        src, idx, iout = ia.src.to(dev), ia.idx.to(dev), ia.out.to(dev)
        iws = dgr.workspace(dgr.index_add_workspace_bytes(262144, 16384, 128), dev)
        ops["index_add"] = lambda iout=iout, src=src, idx=idx, iws=iws: dgr.det_index_add(iout, src, idx, ws=iws)
        host["index_add"] = ([ia.src, ia.idx, ia.out], [src, idx, iout])
        outs["index_add"] = iout
    if with_wgrad and want("wgrad"):
        wi = gi.wgrad_full() if not small else gi.wgrad_input(8, 8192, 4096, 2048, seed=5)
        G, X, offs, mg = wi.G.to(dev), wi.X.to(dev), wi.offs.to(dev), wi.main_grad.to(dev)
        wws = dgr.workspace(dgr.wgrad_workspace_bytes(8, 4096, 2048), dev)
        ops["wgrad"] = (lambda G=G, X=X, offs=offs, mg=mg, wws=wws:
                        dgr.grouped_wgrad_accumulate(G, X, offs, mg, ws=wws))
        host["wgrad"] = ([wi.G, wi.X, wi.offs, wi.main_grad], [G, X, offs, mg])
        outs["wgrad"] = mg
    if want("dbias"):
        db = gi.dbias_full() if not small else gi.dbias_input(16384, 2048, 8, seed=6)
        bdY, boffs, bout = db.dY.to(dev), db.offs.to(dev), db.out.to(dev)
        bws = dgr.workspace(dgr.dbias_workspace_bytes(db.T, db.H, db.E), dev)
        ops["dbias"] = (lambda bdY=bdY, boffs=boffs, bout=bout, bws=bws:
                        dgr.grouped_dbias(bdY, boffs, bout, ws=bws))
        host["dbias"] = ([db.dY, db.offs], [bdY, boffs])
        outs["dbias"] = bout
    if want("topk"):
        tk = gi.topk_full()
        tids, tlg = tk.ids.to(dev), tk.logits.to(dev)
        tout = (torch.empty_like(tids), torch.empty_like(tlg), torch.empty_like(tlg))
        ops["topk"] = lambda tids=tids, tlg=tlg, tout=tout: dgr.topk_canonicalize(tids, tlg, *tout)
        # the inputs (67 MB) fit in L2: the timed calls rotate over copies
        rotations["topk"] = [ops["topk"]] + [
            (lambda tids=tids.clone(), tlg=tlg.clone(), tout=tout: dgr.topk_canonicalize(tids, tlg, *tout))
            for _ in range(ROTATE["topk"] - 1)]
        host["topk"] = ([tk.ids, tk.logits], [tids, tlg])
        outs["topk"] = tout[2]
    if want("aux_loss"):
        ax = gi.aux_full()
        aprobs, atpe = ax.probs.to(dev), ax.tpe.to(dev)
        aout = torch.empty(1, device=dev)
        aws = dgr.workspace(dgr.aux_loss_workspace_bytes(ax.probs.shape[0]), dev)
        ops["aux_loss"] = (lambda aprobs=aprobs, atpe=atpe, aout=aout, aws=aws, sc=ax.scale:
                           dgr.aux_loss(aprobs, atpe, sc, aout, ws=aws))
        # the probabilities (33.5 MB) fit in L2: the timed calls rotate over copies
        rotations["aux_loss"] = [ops["aux_loss"]] + [
            (lambda aprobs=aprobs.clone(), atpe=atpe, aout=aout, aws=aws, sc=ax.scale:
             dgr.aux_loss(aprobs, atpe, sc, aout, ws=aws))
            for _ in range(ROTATE["aux_loss"] - 1)]
        host["aux_loss"] = ([ax.probs, ax.tpe], [aprobs, atpe])
        outs["aux_loss"] = aout
    if want("dsrelu"):
        dsr = gi.dsrelu_full() if not small else gi.dsrelu_input(8, 4096, 2048, 4096, seed=9)
        sA, sB, soffs, sdY = dsr.A.to(dev), dsr.B.to(dev), dsr.offs.to(dev), dsr.dY.to(dev)
        sdp = dsr.dprob.to(dev)
        sws = dgr.workspace(dgr.dsrelu_dprob_workspace_bytes(*dsr.dY.shape), dev)
        ops["dsrelu"] = (lambda sA=sA, sB=sB, soffs=soffs, sdY=sdY, sdp=sdp, sws=sws:
                         dgr.dsrelu_dprob(sA, sB, soffs, sdY, sdp, ws=sws))
        host["dsrelu"] = ([dsr.A, dsr.B, dsr.offs, dsr.dY], [sA, sB, soffs, sdY])
        outs["dsrelu"] = sdp
    steps = ["colsum_large", "colsum_small", "dprob", "colsum_strided", "index_add", "wgrad"]
    order = [n for n in steps + (EXTRAS if only in EXTRAS else []) if n in ops]
    return order, ops, host, outs, rotations


def max_over_ranks(vals: list, device=None) -> list:
    """Element-wise maximum of `vals` over the ranks of the process group (the
    slowest rank's time); the values themselves with one process."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return list(vals)
    if torch.distributed.get_world_size() == 1:
        return list(vals)
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def wgrad_available(dgr) -> bool:
    try:
        import torch
        wi = gi.wgrad_input(1, 16, 128, 256, seed=0)
        dgr.grouped_wgrad_accumulate(wi.G.cuda(), wi.X.cuda(), wi.offs.cuda(), wi.main_grad.cuda())
        torch.cuda.synchronize()
        return True
    except Exception as e:  # noqa: BLE001
        if getattr(e, "code", None) == 2:  # DGR_ERR_UNSUPPORTED: not built yet
            return False
        raise


def run_ours(args, rank, world, local_rank):
    import torch
    import deterministic_gradient_reduction_gb300 as dgr

    dgr.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    with_wgrad = wgrad_available(dgr)
    order, ops, host, outs, rotations = make_ops(dev, torch, dgr, with_wgrad, args.only, args.small)
    if args.only or args.small:  # a profiling run: time it, print the per-operation figures only
        for _ in range(args.warmup):
            for name in order:
                ops[name]()
        torch.cuda.synchronize()
        for _ in range(args.steps):
            for name in order:
                ops[name]()
        torch.cuda.synchronize()
        if rank == 0:
            print(json.dumps({"profile_run": True, "only": args.only, "small": args.small, "ops": order}))
        return
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up
    for _ in range(args.warmup):
        for name in order:
            ops[name]()
    torch.cuda.synchronize()

    # timed: device events around every operation of every step
    K = args.steps
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for n in order}
    step0, step1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local_rank)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    sampler.mark(True)
    step0.record(stream)
    for k in range(K):
        for name in order:
            a, b = ev[name][k]
            a.record(stream)
            ops[name]()
            b.record(stream)
    step1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier()
    total_ms = step0.elapsed_time(step1)
    per_ms = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / K for n in order}

    # The five reductions back to back, K times, between one pair of events:
    # the whole-job time of the reduction work, without the per-operation
    # event records (each bracket above holds a launch and two records, about
    # 4.7 us even around an empty kernel on this GPU).
    red_order = [n for n in order if n in REDUCTIONS]
    for n in red_order:
        ops[n]()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    r0.record(stream)
    for k in range(K):
        for n in red_order:
            ops[n]()
    r1.record(stream)
    torch.cuda.synchronize()
    barrier()
    red_b2b_ms = r0.elapsed_time(r1) / K

    # max over ranks
    if world > 1:
        m = max_over_ranks([total_ms, red_b2b_ms] + [per_ms[n] for n in order], dev)
        total_ms, red_b2b_ms = m[0], m[1]
        per_ms = {n: m[i + 2] for i, n in enumerate(order)}

    # end to end through host buffers: pinned host inputs copied in, outputs read back, every step
    # the next rows of the scope, each timed on its own after the step (not in
    # the step, its value or its launch count). Each is captured as a CUDA graph
    # of 20 calls and the graph replayed, so that the device time of a short
    # call is not hidden behind the host's per-call work (the library holds no
    # host state and synchronises nothing, so its calls capture as they run);
    # plain launches if capture is refused.
    extra_ms, extra_how, extra_win = {}, {}, {}
    for n in [x for x in EXTRAS if x in ops]:
        for _ in range(args.warmup):
            ops[n]()
        torch.cuda.synchronize()
        reps = 20
        graph = None
        try:
            graph = torch.cuda.CUDAGraph()
            calls_n = rotations.get(n, [ops[n]])
            with torch.cuda.graph(graph):
                for r in range(reps):
                    calls_n[r % len(calls_n)]()
            graph.replay()
            torch.cuda.synchronize()
        except Exception:  # noqa: BLE001
            graph = None
            torch.cuda.synchronize()
        n_rep = max(1, K // reps) if graph is not None else K
        if graph is not None and args.next_min_s > 0:  # long enough for its clocks to be sampled
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            n_rep = min(5000, max(n_rep, int(1000.0 * args.next_min_s / max(e0.elapsed_time(e1), 1e-3)) + 1))
        evx = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
        barrier()
        torch.cuda.synchronize()
        tx0 = time.time()
        for a, b in evx:
            a.record(stream)
            if graph is not None:
                graph.replay()
            else:
                ops[n]()
            b.record(stream)
        torch.cuda.synchronize()
        extra_win[n] = (tx0, time.time())
        calls = n_rep * (reps if graph is not None else 1)
        extra_ms[n] = sum(a.elapsed_time(b) for a, b in evx) / calls
        extra_how[n] = f"CUDA graph of {reps} calls, {n_rep} replays" if graph is not None else "plain launches"
        if world > 1:
            extra_ms[n] = max_over_ranks([extra_ms[n]], dev)[0]

    clocks = sampler.stop()  # the step's window
    extra_clocks = {n: sampler.window(*w) for n, w in extra_win.items()}

    e2e = run_e2e(args, torch, order, ops, host, outs, stream, world, dev)

    if rank != 0:
        return
    peaks = load_peaks()
    traffic = load_traffic()  # per-launch DRAM bytes of the kernels as they stand (profiles/)
    red_ms = sum(per_ms[n] for n in REDUCTIONS)
    red_bytes = sum(ALGO[n] for n in REDUCTIONS)
    value = world * red_bytes / (red_b2b_ms * 1e-3) / 1e9
    value_per_op = world * red_bytes / (red_ms * 1e-3) / 1e9
    parts = {}
    for n in order:
        ms = per_ms[n]
        if n == "wgrad":
            tf = ALGO["wgrad_flop"] / (ms * 1e-3) / 1e12
            pk, pk_name = tensor_peak(peaks, clocks)
            parts[n] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1), "frac_bf16": round(tf / pk, 4),
                        "peak": pk, "peak_name": pk_name, "frac_bf16_burst": round(tf / peaks["bf16"], 4),
                        "frac_bf16_sustained": round(tf / peaks["bf16_sus"], 4), "launches": LAUNCHES[n]}
        else:
            gbs = ALGO[n] / (ms * 1e-3) / 1e9
            parts[n] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm"], 4),
                        "launches": LAUNCHES[n], "dram_traffic": traffic.get(n)}
    next_rows = {}
    for n, ms in extra_ms.items():
        if n == "dsrelu":
            tf = ALGO["dsrelu_flop"] / (ms * 1e-3) / 1e12
            pk, pk_name = tensor_peak(peaks, extra_clocks.get(n))
            next_rows[n] = {"us": round(ms * 1e3, 2), "tflops": round(tf, 1), "frac_bf16": round(tf / pk, 4),
                            "peak": pk, "peak_name": pk_name, "frac_bf16_burst": round(tf / peaks["bf16"], 4),
                            "frac_bf16_sustained": round(tf / peaks["bf16_sus"], 4), "launches": LAUNCHES[n],
                            "workload": EXTRA_WORKLOADS[n], "timed_as": extra_how[n], "clocks": extra_clocks.get(n)}
            continue
        gbs = ALGO[n] / (ms * 1e-3) / 1e9
        next_rows[n] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm"], 4),
                        "launches": LAUNCHES[n], "dram_traffic": traffic.get(n), "workload": EXTRA_WORKLOADS[n],
                        "timed_as": extra_how[n], "clocks": extra_clocks.get(n)}
    dom = max(order, key=lambda n: per_ms[n])
    if dom == "wgrad":
        ach = ALGO["wgrad_flop"] / (per_ms[dom] * 1e-3) / 1e12
        pk, pk_name = tensor_peak(peaks, clocks)
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(ach / pk, 4), "traffic": traffic.get(dom), "kernel": dom,
                "peak_source": f"{peaks['src']} {pk_name}"}
    else:
        ach = ALGO[dom] / (per_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm"], 4), "traffic": traffic.get(dom), "kernel": dom,
                "peak_source": f"{peaks['src']} hbm"}
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "no flush: every step streams > 3 GB, inputs larger than L2",
                   "l2_next_rows": L2_NEXT_ROWS,
                   "parallelism": f"replicas x{world}", "wgrad": "included" if with_wgrad else "not built"},
        "reductions_frac_hbm": round(value / world / peaks["hbm"], 4),
        "reductions_us": {"back_to_back": round(red_b2b_ms * 1e3, 2), "sum_of_brackets": round(red_ms * 1e3, 2),
                          "value_from_brackets": round(value_per_op, 1)},
        "wgrad_tflops": parts.get("wgrad", {}).get("tflops"),
        "parts": parts, "next_rows": next_rows, "roofline": roof, "e2e": e2e, "clocks": clocks,
        "gpu_launches": K * sum(LAUNCHES[n] for n in order),
        "gpu_launches_reductions_loop": K * sum(LAUNCHES[n] for n in order if n in REDUCTIONS),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
        if "wgrad" in host:
            line["cpu_baseline"]["wgrad"] = wgrad_oracle_sample(host["wgrad"][0])
    print(json.dumps(line), flush=True)


def host_link_gbs(torch, pinned, host, order, stream):
    """GB/s of one copy of the largest pinned input to its device tensor, the best of three (untimed
    by the step; None if it cannot be taken)."""
    try:
        n, i = max(((n, i) for n in order for i in range(len(pinned[n]))),
                   key=lambda ni: pinned[ni[0]][ni[1]].numel() * pinned[ni[0]][ni[1]].element_size())
        src, dst = pinned[n][i], host[n][1][i]
        nbytes = src.numel() * src.element_size()
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None or ms < best else best
        return round(nbytes / (best * 1e-3) / 1e9, 1) if best and best > 0 else None
    except Exception:  # a diagnostic only: the e2e value does not depend on it
        return None


def run_e2e(args, torch, order, ops, host, outs, stream, world, dev):
    pinned = {n: [t.pin_memory() for t in host[n][0]] for n in order}
    res_host = {n: torch.empty(outs[n].shape, dtype=outs[n].dtype, pin_memory=True) for n in order}
    h2d = sum(t.numel() * t.element_size() for n in order for t in pinned[n])
    d2h = sum(t.numel() * t.element_size() for t in res_host.values())
    K = max(1, args.e2e_steps)
    link = host_link_gbs(torch, pinned, host, order, stream)
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for n in order}
    torch.cuda.synchronize()
    for k in range(K):
        for n in order:
            a, b = ev[n][k]
            a.record(stream)
            for hsrc, ddst in zip(pinned[n], host[n][1]):
                ddst.copy_(hsrc, non_blocking=True)
            ops[n]()
            res_host[n].copy_(outs[n], non_blocking=True)
            b.record(stream)
    torch.cuda.synchronize()
    per = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / K for n in order}
    if world > 1:
        m = max_over_ranks([per[n] for n in order], dev)
        per = {n: m[i] for i, n in enumerate(order)}
    red_ms = sum(per[n] for n in REDUCTIONS)
    val = world * sum(ALGO[n] for n in REDUCTIONS) / (red_ms * 1e-3) / 1e9
    out = {"value": round(val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": K, "ms_per_step": round(sum(per.values()), 3)}
    if link is not None:
        out["h2d_link_gbs"] = link  # this host's pinned-to-device copy rate, which bounds the value
    if "wgrad" in per:
        out["wgrad_tflops"] = round(ALGO["wgrad_flop"] / (per["wgrad"] * 1e-3) / 1e12, 2)
    return out


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

class OracleWork:
    """The oracle on contiguous slices of each reduction workload."""

    def __init__(self):
        import oracle
        self.o = oracle
        self.cl = gi.colsum_large()
        self.cs = gi.colsum_small()
        self.cst = gi.colsum_strided()
        self.dp = gi.dprob_full()
        self.ia = gi.index_add_full()
        self.bits = {"cl": gi.bits(self.cl.base), "cs": gi.bits(self.cs.base), "cst": gi.bits(self.cst.base),
                     "dy": gi.bits(self.dp.dY).reshape(-1), "y": gi.bits(self.dp.Y).reshape(-1)}

    def run(self, frac: float) -> tuple[float, int]:
        """Run every reduction on `frac` of its workload; returns (seconds, algorithmic bytes)."""
        o, b = self.o, self.bits
        t = time.perf_counter()
        nbytes = 0
        out = np.zeros(64, np.float32)
        tok = max(128, int(8388608 * frac) // 128 * 128)
        o.ordered_colsum(b["cl"], 1, tok, 64, tok * 64, 64, out)
        nbytes += tok * 64 * 2 + 256
        o.ordered_colsum(b["cs"], 1, 2048, 16, 2048 * 16, 16, np.zeros(16, np.float32))
        nbytes += ALGO["colsum_small"]
        rows = max(1, int(65536 * frac))
        o.ordered_rowdot_dprob(b["dy"], b["y"], rows, 4096, 4096, 4096, np.zeros(rows, np.float32))
        nbytes += rows * 4096 * 4 + rows * 4
        o.ordered_colsum(b["cst"], 4, 2048, 64, 2048 * 128, 128, np.zeros(64, np.float32))
        nbytes += ALGO["colsum_strided"]
        n = max(2048, int(262144 * frac))
        outi = np.zeros((16385, 128), np.float32)
        o.det_index_add(outi, 16384, 128, 128, gi.f32(self.ia.src)[:n], 128, self.ia.idx.numpy()[:n], n)
        nbytes += n * (128 * 4 + 4) + 2 * 16385 * 128 * 4
        return time.perf_counter() - t, nbytes


def host_cpu() -> dict:
    """The host's CPU model (lscpu, else /proc/cpuinfo, else the machine type) and its core count."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:  # noqa: BLE001
        model = None
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            model = None
    import platform
    return {"cpu_model": model or platform.machine() or "unknown", "host_cores": os.cpu_count()}


def cpu_baseline(budget_s: float = 15.0) -> dict:
    w = OracleWork()
    t_small, _ = w.run(1 / 256)
    frac = min(1.0, max(1 / 256, budget_s / max(t_small * 256, 1e-3)))
    t, nbytes = w.run(frac)
    return {"value": round(nbytes / t / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", **host_cpu(),
            "sample": f"single-threaded C oracle on {frac:.3f} of each reduction workload "
                      f"(colsum 1 GiB / dprob 1 GiB / index_add prefixes; small ones whole), {t:.1f} s"}


def wgrad_oracle_sample(wgrad_host, budget_s: float = 3.0, seed: int = 5) -> dict:
    """The wgrad oracle on a seeded sample of output elements of the full
    workload (each element: every 512-token chunk of its expert through the
    tensor-core step model, the chunks folded, added to its main_grad value),
    timed and extrapolated to all E*N*K elements."""
    import oracle
    G, X, offs, mg = wgrad_host
    Gb, Xb = gi.bits(G), gi.bits(X)
    o = offs.numpy().astype(np.int64)
    E, N, K = mg.shape
    mgf = mg.numpy().reshape(-1)
    rng = np.random.default_rng(seed)

    def run(n):
        e = rng.integers(0, E, n)
        nn = rng.integers(0, N, n)
        kk = rng.integers(0, K, n)
        old = mgf[(e * N + nn) * K + kk]
        t = time.perf_counter()
        oracle.wgrad_elements(Gb, Xb, o, N, K, e, nn, kk, old)
        return time.perf_counter() - t

    t16 = max(run(16), 1e-6)
    n = int(min(200000, max(16, budget_s / (t16 / 16))))
    t = run(n)
    full_s = t / n * E * N * K
    return {"tflops_extrapolated": round(2.0 * N * K * int(o[-1]) / full_s / 1e12, 9), "elements_timed": n,
            "seconds": round(t, 2), "full_seconds_extrapolated": round(full_s, 1),
            "sample": f"{n} seeded output elements of the full E{E} N{N} K{K} workload, extrapolated to all "
                      f"{E * N * K} (single thread)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = OracleWork()
    t_small, _ = w.run(1 / 256)
    per_step_budget = args.cpu_budget / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1 / 8192, per_step_budget / max(t_small * 256, 1e-3)))
    for _ in range(args.warmup):
        w.run(frac)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        t, nb = w.run(frac)
        tot_t += t
        tot_b += nb
    val = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "n/a (CPU)", "parallelism": "single host thread",
                       "wgrad": "not in the oracle rate"},
            "cpu_baseline": {"value": round(val, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", **host_cpu(),
                             "sample": f"{frac:.5f} of each reduction workload per step"},
            "e2e": {"value": round(val, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--next-min-s", type=float, default=0.4,
                    help="time each next row for at least this long (its clocks are sampled over it); "
                         "0 for short profiling runs")
    ap.add_argument("--only", choices=["colsum_large", "colsum_small", "dprob", "colsum_strided", "index_add",
                                       "wgrad", "dbias", "topk", "aux_loss", "dsrelu"],
                    help="profiling: run one operation only (no JSON bench line)")
    ap.add_argument("--small", action="store_true",
                    help="profiling: colsum 2097152x64, dprob 16384x4096, wgrad T=8192 (same widths)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
