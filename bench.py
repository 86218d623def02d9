#!/usr/bin/env python3
"""Benchmark of the emulated quick-allreduce data path on one GB300 (or N
independent replicas, one per GPU).

One step = one pass of the whole hot path over the largest workload that
fits one GPU: W=8 emulated ranks, fp16, a per-rank tensor of 8192 x 8192
(128 MiB; 1 GiB of inputs per call), N(0,1) with 0.1 % of the elements
scaled by 50 -- a 70B-class tensor-parallel prefill hidden state -- through
every format (FP, FP8, Q8, Q6, Q4, Q8A, Q4A), one-stage and two-stage: 14
calls, every two-stage call also writing its stage-2 payload.  Inputs are
resident in HBM and larger than L2; L2 is also flushed before every timed
call, outside the timed events: a write of at least twice its size, then a
read of a second buffer of that size, so that the flush leaves no dirty
lines to be written back during the timed call.

metric: GB/s per rank-message = sum of per-rank message bytes (n*2) over
the calls / their device time.  The timed region is K replays of a CUDA
graph holding one step (each call preceded by its L2 flush), timed with
CUDA events; the same graph without the qr calls is replayed K times and
its time subtracted.  The JSON line also carries the HBM roofline of the
fused two-stage quantized launches, a read-heavy streaming reference timed
the same way, the oracle's CPU rate on a bounded sample, an end-to-end rate
through the C ABI with host buffers, the tp2 size sweep of vLLM PR #18473's
timing table (W=2, fp16, 4 KiB .. 128 MiB) and the other workloads.

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

from quantized_allreduce_codec_gb300.inputs import (ALL_FORMATS, BF16, DTYPE_NAMES, F16,  # noqa: E402
                                                    FORMAT_NAMES, FP, FP8, Q4, Q4A, Q6, Q8, Q8A,
                                                    from_bits, sweep_sizes_bytes, sweep_workload,
                                                    workloads, Workload)

METRIC = "emulated quick-allreduce GB/s per rank-message and % of HBM roofline, 1×GB300"
HEADLINE = 5  # workloads()[5]: W=8, fp16, 8192 x 8192 per rank, 0.1 % outliers x50
STEP_CALLS = [(f, s) for f in ALL_FORMATS for s in (1, 2)]  # every format, one- and two-stage
TP2_CALLS = [(FP, 1), (FP, 2), (FP8, 2), (Q8, 2), (Q6, 2), (Q4, 2)]  # the tp2 table's kernels
TP2_BYTES = 64 << 20
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


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_W8_fp16_step.txt")


def kernel_sources_sha256() -> str:
    """Hash of the kernel sources the committed ncu traffic was taken on."""
    import hashlib
    h = hashlib.sha256()
    for f in ("qr_device.cuh", "qr_kernels.cu"):
        with open(os.path.join(ROOT, "quantized_allreduce_codec_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def step_routes(qr, W: int, n: int) -> str:
    """The kernel path of each call of the bench step, in step order."""
    return ",".join(str(qr.qr_kernel_path(W, F16, fmt, st, n)) for fmt, st in STEP_CALLS)


def recorded_traffic(routes: str):
    """DRAM bytes per launch per kernel from the committed ncu summary
    (lines key=value), if it was taken on the current kernel sources (matched
    by hash) with every call of the step on the kernel path it takes now;
    else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            fields = dict(ln.strip().split("=", 1) for ln in f if "=" in ln and not ln.startswith("#"))
    except OSError:
        return None
    if fields.get("sources_sha256") != kernel_sources_sha256() or fields.get("step_routes") != routes:
        return None
    return fields


def served_by(qr, W: int, dtype: int, fmt: int, stages: int, n: int) -> str:
    """The kernel that serves a call of this shape (the library's routing;
    stages 0 = qr_quantize)."""
    path = qr.qr_kernel_path(W, dtype, fmt, stages, n)
    if path == qr.PATH_DIRECT:
        if stages == 0:
            return "qr_encode_kernel"
        block = W in (2, 4) and fmt not in (FP, FP8) and n >= (3 << 20 if W == 2 else 4 << 20)
        return "qr_block_kernel" if block else "qr_direct_kernel"
    return "qr_pipeline_kernel"


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def headline_config(wl: Workload, world: int) -> dict:
    """The workload description both arms print (identical keys and values)."""
    return {"workload": f"{wl.name}: W={wl.W} emulated ranks, {DTYPE_NAMES[wl.dtype]}, per-rank tensor "
                        f"[8192 x 8192] ({wl.n} elements, {wl.n * 2 >> 20} MiB), N(0,1) with 0.1% of the "
                        f"elements x50 (seed {1000 * wl.key}+r); one step = {len(STEP_CALLS)} calls: "
                        "FP, FP8, Q8, Q6, Q4, Q8A, Q4A, each one-stage and two-stage (two-stage calls write "
                        "their stage-2 payload)",
            "W": wl.W, "dtype": DTYPE_NAMES[wl.dtype], "per_rank_elems": wl.n, "per_rank_bytes": wl.n * 2,
            "calls_per_step": len(STEP_CALLS),
            "l2": "inputs (W x 128 MiB per call) larger than the 126 MiB L2; on the GPU, L2 also flushed before "
                  "every timed call, outside the timed events (a 256 MiB write, then a 256 MiB read of a "
                  "second buffer)",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU, W ranks emulated in HBM"}


def workload_inputs(wl: Workload) -> list:
    """The workload's rank messages (uint16 bits), ranks drawn in parallel
    host threads (each rank has its own seeded generator)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(wl.W, host_threads())) as ex:
        return list(ex.map(wl.rank_bits, range(wl.W)))


def sample_block_elems(n: int, count: int, seed: int) -> np.ndarray:
    """Element indices of `count` distinct 32-element blocks, sorted."""
    rng = np.random.default_rng(seed)
    blocks = np.sort(rng.choice(n // 32, min(count, n // 32), replace=False))
    return (blocks[:, None] * 32 + np.arange(32)[None, :]).reshape(-1)


class GpuTimer:
    """Device time of a sequence of calls: CUDA graphs of [L2 flush, call]
    pairs replayed and timed with CUDA events on the replaying stream, minus
    the same graph of flushes alone."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        props = torch.cuda.get_device_properties(dev)
        self.l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
        self.flush_buf = torch.empty(max(2 * self.l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
        self.clean_buf = torch.ones(self.flush_buf.numel(), dtype=torch.float32, device=dev)
        self.cap_stream = torch.cuda.Stream(device=dev)
        self.flush_graphs = {}

    def flush(self):
        # write more than twice the L2 (evicts the inputs), then read a second
        # buffer of that size so the dirty lines of the write are written back
        # here rather than inside the next timed call
        self.flush_buf.fill_(1)
        self.clean_buf.sum()

    def capture(self, fn):
        g = self.torch.cuda.CUDAGraph()
        self.torch.cuda.synchronize()
        with self.torch.cuda.graph(g, stream=self.cap_stream):
            fn()
        self.torch.cuda.synchronize()
        return g

    def replay_time(self, g, reps):
        torch = self.torch
        s = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(reps):
            g.replay()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3

    def per_call_seconds(self, fn, reps, pairs=7):
        """Device time of fn per call: [flush, fn] x reps minus [flush] x reps.
        The two graphs are replayed in turn `pairs` times and the median of
        the paired differences is taken: the flush dominates every replay,
        so a single difference carries the flush's run-to-run jitter (about
        a tenth of a 10 us call)."""
        fn()  # eager first call: any one-time set-up happens outside capture
        self.torch.cuda.synchronize()
        g1 = self.capture(lambda: [(self.flush(), fn()) for _ in range(reps)])
        if reps not in self.flush_graphs:
            self.flush_graphs[reps] = self.capture(lambda: [self.flush() for _ in range(reps)])
        g0 = self.flush_graphs[reps]
        for g in (g1, g0):
            g.replay()
        diffs = []
        for _ in range(pairs):
            t1 = self.replay_time(g1, 1)
            diffs.append(t1 - self.replay_time(g0, 1))
        del g1
        return max(statistics.median(diffs) / reps, 1e-9)


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
    timer = GpuTimer(dev)
    flush = timer.flush

    wl = workloads()[HEADLINE]
    n, W = wl.n, wl.W
    host = workload_inputs(wl)
    ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in host]
    out = torch.empty(n, dtype=torch.int16, device=dev)
    wires = {f: torch.empty(encoded_bytes(f, n), dtype=torch.uint8, device=dev) for f in ALL_FORMATS}

    def call(fmt, stages):
        # stream=None: torch's current stream (the capture stream inside a graph)
        qr.qr_allreduce_emulated(W, wl.dtype, fmt, stages, ins, n, out, wires[fmt] if stages == 2 else None, None)

    # warm-up, eager (also first-call set-up of every instantiation used)
    for _ in range(args.warmup):
        for fmt, st in STEP_CALLS:
            flush()
            call(fmt, st)
    torch.cuda.synchronize()
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised during warm-up")

    # The timed work runs as CUDA-graph replays: one step = the 14 calls, each
    # preceded by an L2 flush.  A second graph holds the same flushes and
    # nothing else; its time is subtracted, so the reported time is the qr
    # kernels' device time with launch latency overlapped as in any stream of
    # work.
    step_graph = timer.capture(lambda: [(flush(), call(fmt, st)) for fmt, st in STEP_CALLS])
    flush_graph = timer.capture(lambda: [flush() for _ in STEP_CALLS])
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
    t_steps = timer.replay_time(step_graph, K)          # K timed steps (synchronised on both sides)
    wall = time.perf_counter() - wall0
    dist_barrier()
    clocks = sampler.stop()
    t_flush = timer.replay_time(flush_graph, K)         # the same flushes alone
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised in the timed region")
    my_total = t_steps - t_flush
    max_total = dist_max(my_total, dev)
    step_bytes = sum(n * 2 for _ in STEP_CALLS)
    value = aggregate(K * step_bytes, max_total, world)
    del step_graph, flush_graph

    # per-call device times (graphs) and eager event times, for the breakdown
    peak, peak_kind = read_peaks()
    per_format = {}
    q2_bytes = q2_time = all_bytes = all_time = 0.0
    stream = torch.cuda.current_stream()
    for fmt, st in STEP_CALLS:
        b = bytes_alg(W, n, fmt, st, st == 2)
        t = timer.per_call_seconds(lambda: call(fmt, st), args.graph_reps)
        eager = []
        for it in range(args.warmup + args.eager_iters):
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
        all_bytes += b
        all_time += t
        if fmt != FP and st == 2:
            q2_bytes += b
            q2_time += t
    achieved_q2 = q2_bytes / q2_time / 1e9
    n_q2 = sum(1 for f, st in STEP_CALLS if f != FP and st == 2)
    # the step's launches grouped by the kernel the library routes them to;
    # the roofline describes the kernel with the largest share of the time
    kernels = {}
    for fmt, st in STEP_CALLS:
        k = kernels.setdefault(served_by(qr, W, wl.dtype, fmt, st, n), {"launches": 0, "bytes": 0.0, "seconds": 0.0,
                                                                          "calls": []})
        k["launches"] += 1
        k["bytes"] += bytes_alg(W, n, fmt, st, st == 2)
        k["seconds"] += per_format[step_name(fmt, st)]["us"] * 1e-6
        k["calls"].append(step_name(fmt, st))
    dominant = max(kernels, key=lambda name: kernels[name]["seconds"])
    dk = kernels[dominant]
    achieved = dk["bytes"] / dk["seconds"] / 1e9
    kernel_shares = {name: {"launches": v["launches"], "share_of_step_time": round(v["seconds"] / all_time, 3),
                            "achieved_GBps": round(v["bytes"] / v["seconds"] / 1e9, 1),
                            "frac_of_measured_peak": round(v["bytes"] / v["seconds"] / 1e9 / peak, 4),
                            "calls": v["calls"]} for name, v in kernels.items()}

    # ---------------- a W:1 streaming reference ----------------
    # The measured copy peak moves reads and writes 1:1; these calls read W
    # streams for about one written, a mix HBM serves faster.  The library's
    # FP one-stage call on the same inputs is exactly such a stream with no
    # codec (W reads, binary32 adds, one write), timed the same way: the
    # dominant kernel is also reported against its rate.
    fp1 = per_format[step_name(FP, 1)]
    w_to_1 = {"GBps": fp1["hbm_GBps"], "us": fp1["us"],
              "how": f"FP one-stage on the same inputs: {W} streams read, 1 written, binary32 adds, no codec",
              "dominant_frac_of_it": round(achieved / fp1["hbm_GBps"], 4),
              "two_stage_quantized_frac_of_it": round(achieved_q2 / fp1["hbm_GBps"], 4)}

    # ---------------- deviation from the exact sum, per format (rank 0) ----------------
    errors = {}
    if rank == 0 and not args.no_extras:
        idx = sample_block_elems(n, 1 << 15, 5)
        sub = [h[idx] for h in host]
        for fmt, st in STEP_CALLS:
            call(fmt, st)
            torch.cuda.synchronize()
            got = out.cpu().numpy().view(np.uint16)[idx]
            errors[step_name(fmt, st)] = error_vs_exact(sub, got, wl.dtype, fmt, st)
        errors["sample"] = f"{idx.size // 32} random blocks ({idx.size} elements) of the message"
    traffic = recorded_traffic(step_routes(qr, W, n))
    t_key = f"{dominant}.bytes_per_launch"
    roofline = {"kernel": f"{dominant} (W={W}, fp16, 128 MiB per rank; {dk['launches']} of the step's "
                          f"{len(STEP_CALLS)} launches, routed to it by the measured kernel-path table: "
                          f"{', '.join(dk['calls'])})",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_of_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": (float(traffic[t_key]) if traffic and t_key in traffic else None),
                "algorithmic_bytes_per_launch": round(dk["bytes"] / dk["launches"]),
                "traffic_note": (traffic.get("note") if traffic and t_key in traffic
                                 else "no ncu capture of the current kernel sources"),
                "timing": f"per-call device time from CUDA-graph replays ({args.graph_reps} calls, "
                          "flush-only graph subtracted); achieved = the kernel's algorithmic bytes over its "
                          "launches / their summed time",
                "kernels": kernel_shares,
                "two_stage_quantized": {"achieved_GBps": round(achieved_q2, 1),
                                        "frac": round(achieved_q2 / peak, 4), "launches": n_q2},
                "step_achieved_all_14_launches": round(all_bytes / all_time / 1e9, 1),
                "step_frac_all_14_launches": round(all_bytes / all_time / 1e9 / peak, 4),
                "w_to_1_stream": w_to_1}

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
                   f"its output back, in chunks of {chunk} elements whose copies overlap the kernels (the "
                   "stage-2 payload stays on the device)"}
    del pin_in, pin_out, workspace

    # ---------------- the headline workload through the staged path ----------------
    extra = {}
    if not args.no_extras:
        st1 = torch.empty(qr.qr_stage1_bytes(W, Q8, n), dtype=torch.uint8, device=dev)
        res = {}
        for fmt in (Q8, Q4):
            t = timer.per_call_seconds(lambda: qr.qr_allreduce_staged(W, wl.dtype, fmt, ins, n, out, wires[fmt],
                                                                      st1), args.sweep_reps)
            ba = bytes_alg_staged(W, n, fmt)
            res[f"{FORMAT_NAMES[fmt]}-2stage-staged"] = {
                "us": round(t * 1e6, 1), "fused_us": per_format[step_name(fmt, 2)]["us"],
                "algbw_GBps": round(n * 2 / t / 1e9, 1), "hbm_GBps": round(ba / t / 1e9, 1),
                "hbm_frac": round(ba / t / 1e9 / peak, 3)}
        extra[wl.name + " staged"] = res
        del st1
    del ins, out, wires
    torch.cuda.empty_cache()

    # ---------------- tp2 size sweep (the timing table's sizes, then 128 MiB) ----------------
    sweep, codec, staged = {}, {}, {}
    if not args.no_extras:
        tp2 = sweep_workload(TP2_BYTES)
        tp2_host = workload_inputs(tp2)
        t_ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in tp2_host]
        t_out = torch.empty(tp2.n, dtype=torch.int16, device=dev)
        t_wires = {f: torch.empty(encoded_bytes(f, tp2.n), dtype=torch.uint8, device=dev) for f, _ in TP2_CALLS}

        def sweep_point(nn, sub, o, wdict):
            row = {}
            for fmt, st in TP2_CALLS:
                t = timer.per_call_seconds(
                    lambda: qr.qr_allreduce_emulated(2, F16, fmt, st, sub, nn, o, wdict[fmt] if st == 2 else None,
                                                     None), args.sweep_reps)
                row[step_name(fmt, st)] = {"us": round(t * 1e6, 2),
                                           "hbm_frac": round(bytes_alg(2, nn, fmt, st, st == 2) / t / 1e9 / peak, 3)}
            return row

        for size in sweep_sizes_bytes():
            nn = size // 2
            sweep[str(size)] = sweep_point(nn, [t[:nn] for t in t_ins], t_out, t_wires)
        big = sweep_workload(128 << 20)
        big_ins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in workload_inputs(big)]
        big_out = torch.empty(big.n, dtype=torch.int16, device=dev)
        big_wires = {f: torch.empty(encoded_bytes(f, big.n), dtype=torch.uint8, device=dev) for f, _ in TP2_CALLS}
        sweep[str(128 << 20)] = sweep_point(big.n, big_ins, big_out, big_wires)
        del big_ins, big_out, big_wires
        torch.cuda.empty_cache()

        # ---------------- the codec on its own (qr_quantize / qr_dequantize) ----------------
        src = t_ins[0]
        nn = tp2.n
        for fmt in (FP8, Q8, Q6, Q4, Q8A, Q4A):
            enc = torch.empty(encoded_bytes(fmt, nn), dtype=torch.uint8, device=dev)
            qr.qr_quantize(F16, fmt, src, nn, enc)
            row = {}
            for name, fn in (("quantize", lambda: qr.qr_quantize(F16, fmt, src, nn, enc)),
                             ("dequantize", lambda: qr.qr_dequantize(F16, fmt, enc, nn, t_out))):
                t = timer.per_call_seconds(fn, args.sweep_reps)
                ba = nn * 2 + encoded_bytes(fmt, nn)
                row[name] = {"us": round(t * 1e6, 2), "hbm_GBps": round(ba / t / 1e9, 1),
                             "hbm_frac": round(ba / t / 1e9 / peak, 3)}
            codec[FORMAT_NAMES[fmt]] = row
            del enc

        # ---------------- staged two-stage path, tp2 64 MiB ----------------
        st1 = torch.empty(max(qr.qr_stage1_bytes(2, f, nn) for f in (FP8, Q8, Q6, Q4)), dtype=torch.uint8,
                          device=dev)
        for fmt in (FP8, Q8, Q6, Q4):
            t_fused = timer.per_call_seconds(
                lambda: qr.qr_allreduce_emulated(2, F16, fmt, 2, t_ins, nn, t_out, t_wires[fmt]), args.sweep_reps)
            t = timer.per_call_seconds(lambda: qr.qr_allreduce_staged(2, F16, fmt, t_ins, nn, t_out, t_wires[fmt],
                                                                      st1), args.sweep_reps)
            ba = bytes_alg_staged(2, nn, fmt)
            staged[FORMAT_NAMES[fmt]] = {"us": round(t * 1e6, 2), "fused_us": round(t_fused * 1e6, 2),
                                         "hbm_GBps": round(ba / t / 1e9, 1),
                                         "hbm_frac": round(ba / t / 1e9 / peak, 3)}
        del st1, t_ins, t_out, t_wires
        torch.cuda.empty_cache()

        # ---------------- the other workloads ----------------
        for key in (3, 4):
            w = workloads()[key]
            host_w = workload_inputs(w)
            dins = [torch.from_numpy(x.view(np.int16)).to(dev) for x in host_w]
            o = torch.empty(w.n, dtype=torch.int16, device=dev)
            res = {}
            for fmt in w.formats:
                wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
                for st in w.stages:
                    t = timer.per_call_seconds(
                        lambda: qr.qr_allreduce_emulated(w.W, w.dtype, fmt, st, dins, w.n, o,
                                                         wire if st == 2 else None, None),
                        args.sweep_reps)
                    ba = bytes_alg(w.W, w.n, fmt, st, st == 2)
                    res[step_name(fmt, st)] = {"us": round(t * 1e6, 1),
                                               "algbw_GBps": round(w.n * 2 / t / 1e9, 1),
                                               "hbm_GBps": round(ba / t / 1e9, 1),
                                               "hbm_frac": round(ba / t / 1e9 / peak, 3),
                                               "frac_of_nominal_8TBps": round(ba / t / 1e9 / NOMINAL_HBM_GBS, 3)}
                del wire
            # the bf16 -> fp16 cast option against native bf16: speed, and
            # error against the exact sum on 4096 sampled blocks
            idx = sample_block_elems(w.n, 4096, key)
            exact = sum(from_bits(h[idx], BF16).astype(np.float64) for h in host_w)
            for fmt in w.formats:
                wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
                row = {}
                for tag, dt in (("native_bf16", BF16), ("cast_via_fp16", 2)):
                    t = timer.per_call_seconds(
                        lambda: qr.qr_allreduce_emulated(w.W, dt, fmt, 2, dins, w.n, o, wire, None),
                        args.sweep_reps)
                    got = from_bits(o.cpu().numpy().view(np.uint16)[idx], BF16).astype(np.float64)
                    err = np.abs(got - exact)
                    row[tag] = {"us": round(t * 1e6, 1), "max_abs_err": float(err.max()),
                                "mean_abs_err": float(err.mean()), "inf_outputs": int(np.isinf(got).sum())}
                res[f"{FORMAT_NAMES[fmt]}-2stage-cast-option"] = row
                del wire
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
            "timing": f"K replays of a CUDA graph holding one step ({len(STEP_CALLS)} [L2 flush, qr call] pairs), "
                      "timed with CUDA events, minus K replays of the same graph without the qr calls",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": headline_config(wl, world),
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
    of wall time over the step's calls: on every host core (block runs
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
    wl = workloads()[HEADLINE]
    m = min(args.ref_elems, wl.n)
    m -= m % 32
    host = [x[:m].copy() for x in workload_inputs(wl)]
    T = host_threads()
    for _ in range(args.warmup):
        oracle_step(wl.dtype, host, T)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl.dtype, host, T)
    t = time.perf_counter() - t0
    value = args.steps * len(STEP_CALLS) * m * 2 / t / 1e9
    sample = (f"each step runs all {len(STEP_CALLS)} calls of the step on the first {m} elements "
              f"({m * 2 >> 10} KiB, {m // 32} blocks) of each rank's message, split into whole-block runs on "
              f"{T} host threads; the result is defined block by block, so the rate per rank-message byte "
              "is that of the whole message")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": headline_config(wl, world),
        "cpu_baseline": {"kind": "oracle", "cores": T, "value": round(value, 6), "unit": "GB/s",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "the reference arm is the repository's CPU oracle (no reference implementation ships "
                "with the source pages), timed on a bounded sample of the same workload: " + sample,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# kernel-path selection sweep (writes the measurements the routing table is
# generated from: quantized_allreduce_codec_gb300/select_table.py)
# ----------------------------------------------------------------------------
def select_grid_bytes() -> list:
    """Per-rank message sizes of the selection sweep: powers of two from 4 KiB
    to 128 MiB, plus the midpoints 1.5 MiB, 3 MiB, ..., 96 MiB where the
    kernels' times cross."""
    return sorted([4096 << k for k in range(16)] + [3 << (19 + k) for k in range(7)])


def run_select_sweep(args):
    import torch

    import quantized_allreduce_codec_gb300 as qr
    from quantized_allreduce_codec_gb300 import build as qr_build

    qr_build.build()
    qr.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    timer = GpuTimer(dev)
    grid = select_grid_bytes()
    maxn = grid[-1] // 2
    gen = torch.Generator(device=dev)
    records = []
    t_start = time.time()
    for dt in (F16, BF16, 2):
        for W in (1, 2, 4, 8):
            gen.manual_seed(7000 + 10 * dt + W)
            ins = []
            for _ in range(W):  # N(0,1) with 0.1 % of the elements x50, as the LLM-like workloads
                x = torch.randn(maxn, device=dev, generator=gen)
                x[torch.rand(maxn, device=dev, generator=gen) < 0.001] *= 50
                ins.append(x.to(torch.float16 if dt == F16 else torch.bfloat16).view(torch.int16).contiguous())
                del x
            out = torch.empty(maxn, dtype=torch.int16, device=dev)
            wire = torch.empty(encoded_bytes(FP, maxn), dtype=torch.uint8, device=dev)
            for mode in (0, 1, 2):
                if mode == 0 and (W != 1 or dt == 2):
                    continue
                for fmt in ALL_FORMATS:
                    for size in grid:
                        n = size // 2
                        sub = [x[:n] for x in ins]
                        if mode == 0:
                            fn = lambda: qr.qr_quantize(dt, fmt, sub[0], n, wire)  # noqa: E731
                        else:
                            fn = lambda: qr.qr_allreduce_emulated(W, dt, fmt, mode, sub, n, out,  # noqa: E731
                                                                  wire if mode == 2 else None)
                        reps = 20 if size <= (1 << 20) else 10 if size <= (16 << 20) else 5
                        rec = {"dt": dt, "mode": mode, "W": W, "fmt": fmt, "n": n}
                        paths = [("direct", qr.PATH_DIRECT), ("pipeline", qr.PATH_PIPELINE)]
                        if W <= 4:  # narrow tiles are built for W <= 4
                            paths.append(("narrow", qr.PATH_PIPELINE_NARROW))
                        for name, path in paths:
                            with qr.forced_kernel_path(path):
                                rec[f"us_{name}"] = round(timer.per_call_seconds(fn, reps) * 1e6, 3)
                        records.append(rec)
            del ins, out, wire
            torch.cuda.empty_cache()
            print(f"select sweep: dtype {dt} W {W} done ({time.time() - t_start:.0f} s)", file=sys.stderr, flush=True)
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised in the selection sweep")
    props = torch.cuda.get_device_properties(dev)
    doc = {"device": props.name, "sms": props.multi_processor_count,
           "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()),
           "how": "per call shape (dtype, mode 0 = qr_quantize / 1 = one-stage / 2 = two-stage, W, format) and "
                  "per-rank size n (elements), the device time per call of the direct kernel, the wide-tile "
                  "pipeline and (W <= 4) the narrow-tile pipeline, each forced with qr_set_kernel_path, "
                  "from CUDA-graph replays of [L2 flush, call] "
                  "pairs minus the flushes alone, as in bench.py; inputs N(0,1) with 0.1 % x50 outliers",
           "grid_bytes": grid, "records": records}
    with open(args.select_sweep, "w") as f:
        json.dump(doc, f)
    print(json.dumps({"select_sweep": args.select_sweep, "records": len(records),
                      "seconds": round(time.time() - t_start, 1)}), flush=True)


# ----------------------------------------------------------------------------
# small cases for a profiler (ncu): a few launches each, a few GB at most
# ----------------------------------------------------------------------------
PROFILE_CASES = ("step16M", "w4-bf16-2048x4096-q4a", "codec-32M:FMT", "staged-w2-32M:FMT", "staged-w8-16M:FMT",
                 "tp2-<16|64>MiB:FMT:STAGES")


def run_profile_case(args):
    """Launch one small case for a profiler, then exit.
    step16M[:FMT:STAGES]: the headline step's calls (every format one- and
      two-stage, or the one named) at 16M elements per rank -- a quarter of
      the W=8 8192x8192 workload, 256 MiB of inputs, drawn with the same
      recipe (N(0,1), 0.1 % x50) from torch's generator -- each on the kernel
      the library routes the full-size call to (forced with the override),
      each launched twice (the first launch warms up).
    w4-bf16-2048x4096-q4a: the W=4 bf16 2048x4096 workload's Q4A two-stage
      call on its own inputs, launched three times.
    codec-32M:FMT[:PATH]: qr_quantize then qr_dequantize of a 32M-element
      fp16 N(0,1) message in format FMT, three times each; the encoder the
      library routes to, or the one PATH names (direct, narrow, wide).
    staged-w2-32M:FMT: qr_allreduce_staged, W=2 fp16 N(0,1), 32M elements
      per rank, format FMT, three times.
    staged-w8-16M:FMT: the same at W=8, 16M elements per rank (a quarter of
      the W=8 8192x8192 workload).
    tp2-<16|64>MiB:FMT:STAGES: a size of the tp2 table (W=2 fp16 N(0,1), 16
      or 64 MiB per rank, its seeded inputs), one call three times, routed
      by the library."""
    import torch

    import quantized_allreduce_codec_gb300 as qr
    from quantized_allreduce_codec_gb300 import build as qr_build
    qr_build.build()
    qr.lib()
    dev = torch.device("cuda", 0)
    name, *rest = args.profile_case.split(":")
    done = []
    if name == "step16M":
        W, n, full = 8, 16 << 20, workloads()[HEADLINE].n
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        xs = []
        for _ in range(W):
            x = torch.randn(n, device=dev, generator=g)
            x[torch.rand(n, device=dev, generator=g) < 0.001] *= 50
            xs.append(x.half().view(torch.int16).contiguous())
            del x
        out = torch.empty(n, dtype=torch.int16, device=dev)
        wire = torch.empty(encoded_bytes(FP, n), dtype=torch.uint8, device=dev)
        calls = [(int(rest[0]), int(rest[1]))] if rest else STEP_CALLS
        for fmt, st in calls:
            with qr.forced_kernel_path(qr.qr_kernel_path(W, F16, fmt, st, full)):
                for _ in range(2):
                    qr.qr_allreduce_emulated(W, F16, fmt, st, xs, n, out, wire if st == 2 else None)
            done.append({"call": step_name(fmt, st), "kernel": served_by(qr, W, F16, fmt, st, full)})
    elif name == "w4-bf16-2048x4096-q4a":
        w = workloads()[3]
        xs = [torch.from_numpy(x.view(np.int16)).to(dev) for x in workload_inputs(w)]
        out = torch.empty(w.n, dtype=torch.int16, device=dev)
        wire = torch.empty(encoded_bytes(Q4A, w.n), dtype=torch.uint8, device=dev)
        for _ in range(3):
            qr.qr_allreduce_emulated(w.W, w.dtype, Q4A, 2, xs, w.n, out, wire)
        done.append({"call": "Q4A-2stage", "kernel": served_by(qr, w.W, w.dtype, Q4A, 2, w.n)})
    elif name in ("codec-32M", "staged-w2-32M", "staged-w8-16M") and rest:
        fmt = int(rest[0])
        W, n = (8, 16 << 20) if name == "staged-w8-16M" else (2, 32 << 20)
        g = torch.Generator(device=dev)
        g.manual_seed(6)
        xs = [torch.randn(n, device=dev, generator=g).half().view(torch.int16) for _ in range(W)]
        enc = torch.empty(encoded_bytes(fmt, n), dtype=torch.uint8, device=dev)
        out = torch.empty(n, dtype=torch.int16, device=dev)
        if name == "codec-32M":
            paths = {"direct": qr.PATH_DIRECT, "narrow": qr.PATH_PIPELINE_NARROW, "wide": qr.PATH_PIPELINE}
            path = paths[rest[1]] if len(rest) > 1 else qr.qr_kernel_path(1, F16, fmt, 0, n)
            with qr.forced_kernel_path(path):
                for _ in range(3):
                    qr.qr_quantize(F16, fmt, xs[0], n, enc)
                    qr.qr_dequantize(F16, fmt, enc, n, out)
                kernel = served_by(qr, 1, F16, fmt, 0, n)
            done.append({"call": f"quantize, dequantize {FORMAT_NAMES[fmt]}",
                         "kernel": f"{kernel} ({qr.PATH_NAMES[path]}), qr_decode_kernel"})
        else:
            st1 = torch.empty(qr.qr_stage1_bytes(W, fmt, n), dtype=torch.uint8, device=dev)
            for _ in range(3):
                qr.qr_allreduce_staged(W, F16, fmt, xs, n, out, enc, st1)
            done.append({"call": f"staged W={W} {FORMAT_NAMES[fmt]}",
                         "kernel": "qr_scatter_encode_kernel, qr_owner_reduce_kernel, qr_decode_kernel"})
    elif name in ("tp2-16MiB", "tp2-64MiB") and len(rest) == 2:
        fmt, st = int(rest[0]), int(rest[1])
        w = sweep_workload((16 << 20) if name == "tp2-16MiB" else TP2_BYTES)
        xs = [torch.from_numpy(x.view(np.int16)).to(dev) for x in workload_inputs(w)]
        out = torch.empty(w.n, dtype=torch.int16, device=dev)
        wire = torch.empty(encoded_bytes(fmt, w.n), dtype=torch.uint8, device=dev)
        for _ in range(3):
            qr.qr_allreduce_emulated(2, F16, fmt, st, xs, w.n, out, wire if st == 2 else None)
        done.append({"call": step_name(fmt, st), "kernel": served_by(qr, 2, F16, fmt, st, w.n)})
    else:
        raise SystemExit(f"unknown profile case {args.profile_case!r} (one of {PROFILE_CASES})")
    torch.cuda.synchronize()
    if qr.qr_device_error() != 0:
        raise RuntimeError("kernel wait-limit flag raised")
    print(json.dumps({"profile_case": args.profile_case, "calls": done}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--eager-iters", type=int, default=10)
    ap.add_argument("--graph-reps", type=int, default=20, help="calls per graph for per-call times")
    ap.add_argument("--sweep-reps", type=int, default=10, help="calls per graph in the sweep/extras")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-elems", type=int, default=1 << 20)
    ap.add_argument("--no-extras", action="store_true", help="skip the size sweep and other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", metavar="NAME",
                    help=f"instead of the bench: launch one small case for a profiler ({', '.join(PROFILE_CASES)})")
    ap.add_argument("--select-sweep", metavar="OUT.json",
                    help="instead of the bench: time both kernel paths for every call shape over a size grid "
                         "and write the measurements (the input of select_table.py)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile_case:
        run_profile_case(args)
    elif args.select_sweep:
        run_select_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
