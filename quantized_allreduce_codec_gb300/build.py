"""Build libqr.so in-tree with nvcc for sm_103a.

The per-format kernel file is compiled once per format (-DQR_FMT=<n>) and
the translation units are compiled in parallel, then linked into one shared
library next to this file.  Usage: ``python -m quantized_allreduce_codec_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqr.so")
NUM_FORMATS = 7

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqr.so")
    return path


def _sources():
    return [os.path.join(CSRC, f) for f in ("qr_api.cu", "qr_kernels.cu", "qr_device.cuh", "qr_launch.h",
                                             "qr_staged.cuh", "qr_noalloc.cu", "qr_select_table.h")] + \
        [os.path.join(INCLUDE, "qr.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def _compile(args):
    src, obj, extra, verbose = args
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    jobs = [(os.path.join(CSRC, "qr_api.cu"), os.path.join(BUILD, "qr_api.o"), [], verbose),
            (os.path.join(CSRC, "qr_noalloc.cu"), os.path.join(BUILD, "qr_noalloc.o"), [], verbose)]
    for f in range(NUM_FORMATS):
        jobs.append((os.path.join(CSRC, "qr_kernels.cu"), os.path.join(BUILD, f"qr_kernels_f{f}.o"),
                     [f"-DQR_FMT={f}"], verbose))
    workers = min(len(jobs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        logs = list(ex.map(_compile, jobs))
    if verbose:
        for log in logs:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *[j[1] for j in jobs]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
