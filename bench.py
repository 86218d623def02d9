#!/usr/bin/env python3
"""Benchmark of the emulated quick-allreduce data path on one GB300 (or N
independent replicas, one per GPU).

One step = one pass of the whole hot path over the tp2 workload of the vLLM
PR #18473 timing table at its largest size: W=2 emulated ranks, fp16,
64 MiB per rank, N(0,1), in the table's six kernels -- FP one-stage, FP
two-stage, FP8, Q8, Q6 and Q4 two-stage (every two-stage call also writes
its stage-2 payload).  Inputs are resident in HBM; L2 is flushed before every timed call,
outside the timed events: a write of at least twice its size, then a read
of a second buffer of that size, so that the flush leaves no dirty lines to
be written back during the timed call.

metric: GB/s per rank-message = sum of per-rank message bytes (n*2) over
the calls / their device time.  The timed region is K replays of a CUDA
graph holding one step (each call preceded by its L2 flush), timed with
CUDA events; the same graph without the qr calls is replayed K times and
its time subtracted.  Eager per-call event times are reported beside it
(they include a ~4 us launch gap that even an empty kernel shows).  The JSON line also carries the HBM roofline of the fused
two-stage quantized kernel, the oracle's CPU rate on a bounded sample, an
end-to-end rate through the C ABI with host buffers, a size sweep, and the
other workloads.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 is launched with torchrun; each rank runs the same workload on its
own GPU (replicas: the emulated path has no inter-GPU exchange).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_allreduce_codec_gb300.inputs import (BF16, F16, FORMAT_NAMES, FP, FP8, Q4,  # noqa: E402
                                                    Q4A, Q6, Q8, Q8A, from_bits, sweep_sizes_bytes,
                                                    sweep_workload, workloads, Workload)

METRIC = "emulated quick-allreduce GB/s per rank-message and % of HBM roofline, 1×GB300"
STEP_CALLS = [(FP, 1), (FP, 2), (FP8, 2), (Q8, 2), (Q6, 2), (Q4, 2)]  # the tp2 table's kernels
BENCH_BYTES = 64 << 20
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CODE_BITS = {Q8: 8, Q6: 6, Q4: 4, FP8: 8, Q8A: 8, Q4A: 4}


def encoded_bytes(fmt: int, n: int) -> int:
    if fmt == FP:
        return 2 * n
    nb = (n + 31) // 32
    return nb * (32 * CODE_BITS[fmt] // 8 + (4 if fmt in (Q8A, Q4A) else 2))


def bytes_alg(W: int, n: int, fmt: int, stages: int, wire: bool) -> int:
    """Algorithmic bytes of one emulated allreduce: read W messages, write the
    output, plus the stage-2 payload when it is written."""
    b = W * n * 2 + n * 2
    if stages == 2 and wire:
        b += encoded_bytes(fmt, n)
    return b


def bytes_alg_staged(W: int, n: int, fmt: int) -> int:
    """Algorithmic bytes of the staged (stage-1 materialised) two-stage
    allreduce: encode W messages into the exchange buffer, the owners read it
    back and write the payload, the payload is decoded to the output."""
    c = encoded_bytes(fmt, n)
    return (W + 1) * n * 2 + (2 * W + 2) * c


QMAX = {Q8: 127, Q6: 31, Q4: 7}


def error_vs_exact(host, out_bits, dtype, fmt, stages) -> dict:
    """Deviation of an allreduce output from the fp64 exact sum e of the
    inputs, against the stated bounds: FP within 1 ulp of the dtype; FP8
    within 2^-3 of sum_r |x_r|; a symmetric integer format within
    b1 = sum_r s_r/2 (stage 1, s_r = fp16(max|x_r| / Qmax) per block) plus,
    for two stages, s2/2 with s2 <= (max|e| + b1) / Qmax * (1 + 2^-10) per
    block, plus 1/2 ulp of the dtype and the binary32 summation error.
    Also reported: the largest per-block ratio max|y - e| / max sum_r|x_r|."""
    xs = [from_bits(h, dtype).astype(np.float64) for h in host]
    e = np.sum(xs, axis=0)
    sabs = np.sum([np.abs(x) for x in xs], axis=0)
    y = from_bits(out_bits, dtype).astype(np.float64)
    nb = e.size // 32
    m = nb * 32
    err = np.abs(y - e)[:m]
    mant = 10 if dtype == F16 else 7
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(e[:m]), 2.0 ** -24))) - mant)
    blk = lambda v: np.repeat(np.abs(v[:m]).reshape(nb, 32).max(axis=1), 32)  # noqa: E731
    res = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
           "max_block_rel": float((blk(err) / np.maximum(blk(sabs), 1e-300)).max())}
    if fmt == FP:
        bound = ulp
    elif fmt == FP8:
        bound = 2.0 ** -3 * sabs[:m] + ulp
    elif fmt in QMAX:
        q = QMAX[fmt]
        b1 = np.zeros(m)
        for x in xs:
            b1 += (blk(x) / q).astype(np.float16).astype(np.float64) / 2
        bound = b1 + ulp + 2.0 ** -20 * sabs[:m]
        if stages == 2:
            bound += (blk(e) + blk(b1)) / q * (1 + 2.0 ** -10) / 2
    else:
        return res
    res["within_bound_fraction"] = float(np.mean(err <= bound))
    return res


def step_name(fmt: int, stages: int) -> str:
    return f"{FORMAT_NAMES[fmt]}-{stages}stage"


# ----------------------------------------------------------------------------
# distributed plumbing (replicas) -- host logic, tested with gloo on CPU
# ----------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def dist_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_bytes: float, max_seconds: float, world: int) -> float:
    """Whole-job GB/s: every rank moves per_rank_bytes in at most max_seconds."""
    return world * per_rank_bytes / max_seconds / 1e9


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str, interval_ms: int = 50):
        self.index, self.interval = index, interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, flag in zip(names, parts[4:8]):
                if flag.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def smi_device_id(props, local: int) -> str:
    """nvidia-smi -i selector of this process's GPU (UUID, else PCI bus id,
    else the CUDA index)."""
    uuid = getattr(props, "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    bus = getattr(props, "pci_bus_id", None)
    if bus is not None:
        return f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    return str(local)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel_source: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (matched by hash); else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "qr_pipeline_traffic.txt")
    try:
        fields = dict(ln.split("=", 1) for ln in open(path).read().split() if "=" in ln)
        src = open(kernel_source, "rb").read()
        if fields.get("source_sha256") != hashlib.sha256(src).hexdigest():
            return None
        return fields
    except OSError:
        return None


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_ours(args):
    import torch

    import quantized_allreduce_codec_gb300 as qr
    from quantized_allreduce_codec_gb300 import build as qr_build

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    if rank == 0 or not os.path.exists(qr.LIB_PATH):
        qr_build.build()
    dist_barrier()
    qr.lib()
    dev = torch.device("cuda", local)

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    flush_buf = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    clean_buf = torch.ones(flush_buf.numel(), dtype=torch.float32, device=dev)

    def flush():
        # write more than twice the L2 (evicts the inputs), then read a second
        # buffer of that size so the dirty lines of the write are written back
        # here rather than inside the next timed call
        flush_buf.fill_(1)
        clean_buf.sum()

    wl = sweep_workload(BENCH_BYTES)
    n, W = wl.n, wl.W
    host = wl.inputs()
    ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in host]
    out = torch.empty(n, dtype=torch.int16, device=dev)
    wires = {f: torch.empty(encoded_bytes(f, n), dtype=torch.uint8, device=dev) for f, _ in STEP_CALLS}

    def call(fmt, stages, inputs=None, nn=n, o=out):
        # stream=None: torch's current stream (the capture stream inside a graph)
        inputs = ins if inputs is None else inputs
        qr.qr_allreduce_emulated(len(inputs), wl.dtype, fmt, stages, inputs, nn, o,
                                 wires[fmt] if stages == 2 else None, None)

    # warm-up, eager (also first-call set-up of every instantiation used)
    for _ in range(args.warmup):
        for fmt, st in STEP_CALLS:
            flush()
            call(fmt, st)
    torch.cuda.synchronize()
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised during warm-up")

    # The timed work runs as CUDA-graph replays: one step = the six calls, each
    # preceded by an L2 flush.  A second graph holds the same six flushes and
    # nothing else; its time is subtracted, so the reported time is the qr
    # kernels' device time with launch latency overlapped as in any stream of
    # work (eager per-call events, reported beside it, also count the ~4 us
    # launch gap an empty kernel shows between two events).
    cap_stream = torch.cuda.Stream(device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap_stream):
            fn()
        torch.cuda.synchronize()
        return g

    def replay_time(g, reps):
        s = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(reps):
            g.replay()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3

    flush_graphs = {}

    def per_call_seconds(fn, reps):
        """Device time of fn per call: [flush, fn] x reps minus [flush] x reps."""
        fn()  # eager first call: any one-time set-up happens outside capture
        torch.cuda.synchronize()
        g1 = capture(lambda: [(flush(), fn()) for _ in range(reps)])
        if reps not in flush_graphs:
            flush_graphs[reps] = capture(lambda: [flush() for _ in range(reps)])
        g0 = flush_graphs[reps]
        for g in (g1, g0):
            g.replay()
        t1 = replay_time(g1, 2) / 2
        t0 = replay_time(g0, 2) / 2
        del g1
        return max((t1 - t0) / reps, 1e-9)

    step_graph = capture(lambda: [(flush(), call(fmt, st)) for fmt, st in STEP_CALLS])
    flush_graph = capture(lambda: [flush() for _ in STEP_CALLS])
    for _ in range(args.warmup):
        step_graph.replay()
        flush_graph.replay()
    torch.cuda.synchronize()

    K = args.steps
    sampler = ClockSampler(smi_device_id(props, local))
    dist_barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    t_steps = replay_time(step_graph, K)          # K timed steps (synchronised on both sides)
    wall = time.perf_counter() - wall0
    dist_barrier()
    clocks = sampler.stop()
    t_flush = replay_time(flush_graph, K)         # the same flushes alone
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised in the timed region")
    my_total = t_steps - t_flush
    max_total = dist_max(my_total, dev)
    step_bytes = sum(n * 2 for _ in STEP_CALLS)
    value = aggregate(K * step_bytes, max_total, world)

    # per-call device times (graphs) and eager event times, for the breakdown
    peak, peak_kind = read_peaks()
    per_format = {}
    q_bytes = q_time = 0.0
    stream = torch.cuda.current_stream()
    for fmt, st in STEP_CALLS:
        b = bytes_alg(W, n, fmt, st, st == 2)
        t = per_call_seconds(lambda: call(fmt, st), args.graph_reps)
        eager = []
        for it in range(args.warmup + args.sweep_iters):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call(fmt, st)
            e1.record(stream)
            if it >= args.warmup:
                eager.append((e0, e1))
        torch.cuda.synchronize()
        te = float(np.median([x.elapsed_time(y) for x, y in eager])) * 1e-3
        per_format[step_name(fmt, st)] = {
            "us": round(t * 1e6, 2), "us_eager_events": round(te * 1e6, 2),
            "algbw_GBps": round(n * 2 / t / 1e9, 1), "hbm_GBps": round(b / t / 1e9, 1),
            "frac_of_measured_peak": round(b / t / 1e9 / peak, 3)}
        if fmt != FP:
            q_bytes += b
            q_time += t
    achieved = q_bytes / q_time / 1e9

    # ---------------- deviation from the exact sum, per format (rank 0) ----------------
    errors = {}
    if rank == 0 and not args.no_extras:
        for fmt, st in STEP_CALLS:
            call(fmt, st)
            torch.cuda.synchronize()
            errors[step_name(fmt, st)] = error_vs_exact(host, out.cpu().numpy().view(np.uint16), wl.dtype,
                                                         fmt, st)
    traffic = recorded_traffic(os.path.join(ROOT, "quantized_allreduce_codec_gb300", "csrc",
                                            "qr_device.cuh"))
    roofline = {"kernel": "qr_pipeline_kernel (fused two-stage, quantized formats FP8/Q8/Q6/Q4, fp16, W=2)",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_of_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": (float(traffic["bytes_per_launch"]) if traffic else None),
                "algorithmic_bytes_per_launch": round(q_bytes / 4),
                "traffic_note": (traffic.get("note") if traffic else
                                 "no ncu capture of the current kernel source"),
                "timing": f"per-call device time from CUDA-graph replays ({args.graph_reps} calls, "
                          "flush-only graph subtracted)"}

    # ---------------- end to end through the C ABI, host buffers ----------------
    # qr_allreduce_host: page-locked host inputs in, the output back to host
    # memory, chunked through a device workspace so that the copies in both
    # directions overlap the kernels; every byte crosses the host link each
    # call, inside the timed region.
    Ke = max(1, min(args.steps, args.e2e_steps))
    pin_in = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in host]
    pin_out = torch.empty(n, dtype=torch.int16).pin_memory()
    chunk = qr.DEFAULT_HOST_CHUNK
    workspace = qr.host_workspace(W, FP, chunk, device=dev)  # FP's payload is the largest
    stream = torch.cuda.current_stream()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for warm in (True, False):
        torch.cuda.synchronize()
        dist_barrier()
        e_start.record(stream)
        for _ in range(1 if warm else Ke):
            for fmt, st in STEP_CALLS:
                qr.qr_allreduce_host(W, wl.dtype, fmt, st, pin_in, n, pin_out, None, workspace,
                                     chunk_elems=chunk, stream=stream)
        e_end.record(stream)
        torch.cuda.synchronize()
    e2e_t = dist_max(e_start.elapsed_time(e_end) * 1e-3, dev)
    e2e = {"value": round(aggregate(Ke * step_bytes, e2e_t, world), 2), "unit": "GB/s",
           "h2d_bytes_per_step": sum(W * n * 2 for _ in STEP_CALLS),
           "d2h_bytes_per_step": sum(n * 2 for _ in STEP_CALLS), "steps": Ke,
           "note": "qr_allreduce_host on page-locked host buffers: every call copies its W inputs in and "
                   f"its output back, in chunks of {chunk} elements whose copies overlap the kernels (the stage-2 payload stays on "
                   "the device)"}
    del pin_in, pin_out, workspace

    # ---------------- size sweep (tp2 table sizes, then 128 MiB) ----------------
    sweep = {}
    if not args.no_extras:
        default_limit = qr.qr_direct_limit()

        def sweep_point(nn, sub, o, wdict):
            row = {}
            # both kernels are timed at every size (the default routing picks one)
            paths = [("default", default_limit), ("direct", (1 << 64) - 1), ("pipeline", 0)]
            for fmt, st in STEP_CALLS:
                entry = {}
                for pname, limit in paths:
                    qr.qr_set_direct_limit(limit)
                    t = per_call_seconds(
                        lambda: qr.qr_allreduce_emulated(W, wl.dtype, fmt, st, sub, nn, o,
                                                         wdict[fmt] if st == 2 else None, None),
                        args.sweep_reps)
                    if pname == "default":
                        entry.update({"us": round(t * 1e6, 2),
                                      "hbm_frac": round(bytes_alg(W, nn, fmt, st, st == 2) / t / 1e9 / peak, 3)})
                    else:
                        entry[f"us_{pname}"] = round(t * 1e6, 2)
                qr.qr_set_direct_limit(default_limit)
                row[step_name(fmt, st)] = entry
            return row

        for size in sweep_sizes_bytes():
            nn = size // 2
            sweep[str(size)] = sweep_point(nn, [t[:nn] for t in ins], out, wires)
        # one point past the tp2 table: 128 MiB per rank, its own buffers
        big = sweep_workload(128 << 20)
        big_ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in big.inputs()]
        big_out = torch.empty(big.n, dtype=torch.int16, device=dev)
        big_wires = {f: torch.empty(encoded_bytes(f, big.n), dtype=torch.uint8, device=dev) for f, _ in STEP_CALLS}
        sweep[str(128 << 20)] = sweep_point(big.n, big_ins, big_out, big_wires)
        del big_ins, big_out, big_wires
        torch.cuda.empty_cache()

    # ---------------- the codec on its own (qr_quantize / qr_dequantize) ----------------
    codec = {}
    if not args.no_extras:
        src = ins[0]
        for fmt in (FP8, Q8, Q6, Q4, Q8A, Q4A):
            enc = torch.empty(encoded_bytes(fmt, n), dtype=torch.uint8, device=dev)
            qr.qr_quantize(wl.dtype, fmt, src, n, enc)
            row = {}
            for name, fn in (("quantize", lambda: qr.qr_quantize(wl.dtype, fmt, src, n, enc)),
                             ("dequantize", lambda: qr.qr_dequantize(wl.dtype, fmt, enc, n, out))):
                t = per_call_seconds(fn, args.sweep_reps)
                ba = n * 2 + encoded_bytes(fmt, n)
                row[name] = {"us": round(t * 1e6, 2), "hbm_GBps": round(ba / t / 1e9, 1),
                             "hbm_frac": round(ba / t / 1e9 / peak, 3)}
            codec[FORMAT_NAMES[fmt]] = row
            del enc

    # ---------------- staged two-stage path (stage-1 exchange materialised) ----------------
    staged = {}
    if not args.no_extras:
        st1 = torch.empty(max(qr.qr_stage1_bytes(W, f, n) for f in (FP8, Q8, Q6, Q4)), dtype=torch.uint8,
                          device=dev)
        for fmt in (FP8, Q8, Q6, Q4):
            t = per_call_seconds(lambda: qr.qr_allreduce_staged(W, wl.dtype, fmt, ins, n, out, wires[fmt], st1),
                                 args.sweep_reps)
            ba = bytes_alg_staged(W, n, fmt)
            staged[FORMAT_NAMES[fmt]] = {"us": round(t * 1e6, 2),
                                         "fused_us": per_format[step_name(fmt, 2)]["us"],
                                         "hbm_GBps": round(ba / t / 1e9, 1),
                                         "hbm_frac": round(ba / t / 1e9 / peak, 3)}
        del st1

    # ---------------- the other workloads ----------------
    extra = {}
    if not args.no_extras:
        del ins
        torch.cuda.empty_cache()
        for key in (3, 4, 5):
            w = workloads()[key]
            dins = [torch.from_numpy(w.rank_bits(r).view(np.int16)).to(dev) for r in range(w.W)]
            o = torch.empty(w.n, dtype=torch.int16, device=dev)
            res = {}
            for fmt in w.formats:
                wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
                for st in w.stages:
                    t = per_call_seconds(
                        lambda: qr.qr_allreduce_emulated(w.W, w.dtype, fmt, st, dins, w.n, o,
                                                         wire if st == 2 else None, None),
                        args.sweep_reps)
                    ba = bytes_alg(w.W, w.n, fmt, st, st == 2)
                    res[step_name(fmt, st)] = {"us": round(t * 1e6, 1),
                                               "algbw_GBps": round(w.n * 2 / t / 1e9, 1),
                                               "hbm_GBps": round(ba / t / 1e9, 1),
                                               "hbm_frac": round(ba / t / 1e9 / peak, 3)}
                del wire
            if key in (3, 4):
                # the bf16 -> fp16 cast option against native bf16: speed, and
                # error against the exact sum on 4096 sampled blocks
                host_w = [w.rank_bits(r) for r in range(w.W)]
                rng = np.random.default_rng(key)
                blocks = np.sort(rng.choice(w.n // 32, 4096, replace=False))
                idx = (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)
                exact = sum(from_bits(h[idx], BF16).astype(np.float64) for h in host_w)
                for fmt in w.formats:
                    wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
                    row = {}
                    for tag, dt in (("native_bf16", BF16), ("cast_via_fp16", 2)):
                        t = per_call_seconds(
                            lambda: qr.qr_allreduce_emulated(w.W, dt, fmt, 2, dins, w.n, o, wire, None),
                            args.sweep_reps)
                        got = from_bits(o.cpu().numpy().view(np.uint16)[idx], BF16).astype(np.float64)
                        err = np.abs(got - exact)
                        row[tag] = {"us": round(t * 1e6, 1), "max_abs_err": float(err.max()),
                                    "mean_abs_err": float(err.mean()),
                                    "inf_outputs": int(np.isinf(got).sum())}
                    res[f"{FORMAT_NAMES[fmt]}-2stage-cast-option"] = row
                    del wire
            if key == 5:
                st1 = torch.empty(qr.qr_stage1_bytes(w.W, Q8, w.n), dtype=torch.uint8, device=dev)
                for fmt in (Q8, Q4):
                    wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
                    t = per_call_seconds(
                        lambda: qr.qr_allreduce_staged(w.W, w.dtype, fmt, dins, w.n, o, wire, st1),
                        args.sweep_reps)
                    ba = bytes_alg_staged(w.W, w.n, fmt)
                    res[f"{FORMAT_NAMES[fmt]}-2stage-staged"] = {"us": round(t * 1e6, 1),
                                                                 "algbw_GBps": round(w.n * 2 / t / 1e9, 1),
                                                                 "hbm_GBps": round(ba / t / 1e9, 1),
                                                                 "hbm_frac": round(ba / t / 1e9 / peak, 3)}
                    del wire
                del st1
            extra[w.name] = res
            del dins, o
            torch.cuda.empty_cache()
        if qr.qr_device_error() != 0:
            raise RuntimeError("kernel wait-limit flag raised in the extras")

    # ---------------- CPU baseline: the oracle on a bounded sample ----------------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(host, wl.dtype, args.cpu_seconds)
        if not args.no_extras:
            cpu["per_config_GBps"] = oracle_per_config(cpu["cores"])

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(max_total / K * 1e3, 4),
            "timing": "K replays of a CUDA graph holding one step (six [L2 flush, qr call] pairs), "
                      "timed with CUDA events, minus K replays of the same graph without the qr calls",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "tp2 table, largest size: W=2 emulated ranks, fp16, 64 MiB "
                                   "(33554432 elements) per rank, N(0,1) seed 2000+r; one step = "
                                   "FP 1-stage, FP 2-stage, FP8, Q8, Q6, Q4 2-stage (payload written)",
                       "W": W, "per_rank_bytes": n * 2, "calls_per_step": len(STEP_CALLS),
                       "l2": f"flushed before every timed call, outside the timed events: a "
                             f"{flush_buf.numel() * 4 >> 20} MiB write, then a {clean_buf.numel() * 4 >> 20} MiB "
                             "read of a second buffer (no dirty lines left in L2)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, W ranks emulated in HBM"},
            "roofline": roofline, "per_format": per_format, "error_vs_exact_sum": errors,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": K * len(STEP_CALLS),
            "clocks": clocks, "wall_ms_per_step_incl_flush": round(wall / K * 1e3, 3),
            "flush_ms_per_step": round(t_flush / K * 1e3, 4),
            "sweep_W2_fp16": sweep, "codec_fp16_64MiB": codec, "staged_W2_fp16_64MiB": staged,
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    dist_barrier()


def oracle_step(dtype, xs, threads: int, calls=None) -> None:
    """One bench step (the six calls, or `calls`) through the oracle, the
    message split into `threads` contiguous runs of whole 32-element blocks,
    one per host thread.  The oracle is a C library called through ctypes,
    which releases the GIL, and the result is defined block by block, so the
    runs are independent; the oracle itself is unchanged."""
    import oracle
    calls = STEP_CALLS if calls is None else calls
    m = xs[0].size
    nblk = m // 32
    cuts = [(nblk * i // threads) * 32 for i in range(threads)] + [m]
    parts = [(cuts[i], cuts[i + 1]) for i in range(threads) if cuts[i + 1] > cuts[i]]

    def one(lo_hi):
        lo, hi = lo_hi
        for fmt, st in calls:
            oracle.allreduce(dtype, fmt, st, [x[lo:hi] for x in xs])

    if len(parts) == 1:
        one(parts[0])
        return
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        list(ex.map(one, parts))


def oracle_per_config(threads: int, m: int = 1 << 20) -> dict:
    """The oracle on each of the five workloads' recipes at a bounded size
    (min(n, m) elements per rank, same generator, shape and value mix), per
    format and stage count, on `threads` host threads: GB/s per
    rank-message."""
    import oracle
    oracle.build()
    res = {}
    for w in workloads().values():
        mm = min(w.n, m)
        small = Workload(w.key, w.name, w.W, w.dtype, mm, w.kind, w.formats, w.stages,
                         rows=w.rows if (w.rows and mm % w.rows == 0) else None, sigma=w.sigma)
        xs = small.inputs()
        row = {}
        for fmt in w.formats:
            for st in w.stages:
                t0 = time.perf_counter()
                oracle_step(w.dtype, xs, threads, [(fmt, st)])
                t = time.perf_counter() - t0
                row[step_name(fmt, st)] = round(mm * 2 / t / 1e9, 5)
        res[f"{w.name} (first {mm} elements per rank)"] = row
    return res


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_baseline(host, dtype, seconds: float) -> dict:
    """The oracle on a prefix of the bench workload sized to about `seconds`
    of wall time over the step's six calls: on every host core (block runs
    in parallel threads), and on one core for comparison."""
    import oracle
    oracle.build()
    T = host_threads()

    def run(m, threads):
        t0 = time.perf_counter()
        oracle_step(dtype, [x[:m] for x in host], threads)
        return time.perf_counter() - t0

    probe = 1 << 15
    tp = run(probe, 1)
    m1 = int(min(host[0].size, max(probe, probe * seconds / 2 / max(tp, 1e-6))))
    m1 -= m1 % 32
    t1 = run(m1, 1)
    mT = int(min(host[0].size, m1 * T))
    mT -= mT % 32
    tT = run(mT, T)
    gb = lambda m, t: round(len(STEP_CALLS) * m * 2 / t / 1e9, 5)  # noqa: E731
    return {"value": gb(mT, tT), "unit": "GB/s", "cores": T, "kind": "oracle",
            "single_thread_value": gb(m1, t1),
            "sample": f"first {mT} elements ({mT * 2 / 2**20:.1f} MiB) of each rank's message, all "
                      f"{len(STEP_CALLS)} calls of one step, split into {T} block runs on {T} threads "
                      f"({tT:.1f} s); single-threaded: first {m1} elements ({t1:.1f} s)"}


# ----------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ----------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = sweep_workload(BENCH_BYTES)
    m = args.ref_elems
    host = [wl.rank_bits(r)[:m] for r in range(wl.W)]
    T = host_threads()
    for _ in range(args.warmup):
        oracle_step(wl.dtype, host, T)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl.dtype, host, T)
    t = time.perf_counter() - t0
    value = args.steps * len(STEP_CALLS) * m * 2 / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "tp2 table, largest size: W=2 emulated ranks, fp16, 64 MiB per rank, "
                               "N(0,1); one step = FP 1-stage, FP 2-stage, FP8, Q8, Q6, Q4 2-stage; "
                               f"each step runs the CPU oracle on the first {m} elements of each rank, "
                               f"split into block runs on {T} host threads",
                   "W": wl.W, "per_rank_bytes": wl.n * 2},
        "cpu_baseline": {"kind": "oracle", "cores": T, "value": round(value, 6), "unit": "GB/s",
                         "sample": f"first {m} elements of each rank's message per call, "
                                   f"in {T} block runs on {T} threads"},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the reference arm is the repository's CPU oracle (no reference implementation ships "
                "with the source pages)",
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--sweep-iters", type=int, default=20)
    ap.add_argument("--graph-reps", type=int, default=50, help="calls per graph for per-call times")
    ap.add_argument("--sweep-reps", type=int, default=10, help="calls per graph in the sweep/extras")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-elems", type=int, default=1 << 18)
    ap.add_argument("--no-extras", action="store_true", help="skip the size sweep and other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
