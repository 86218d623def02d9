"""CPU oracle for the quick-allreduce codec and the emulated allreduce.

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``qro.c`` (plain C,
binary32 IEEE operations, contraction off); this module builds it with gcc
and wraps it with ctypes and numpy.  Only the tests, the package's smoke
check and the benchmark's CPU-baseline leg may import this module.  It
imports nothing from the CUDA library and the CUDA library imports nothing
from here.

Parity status: every exported function is pinned by the ``-m "not gpu"``
tests (library casts, brute-force code enumeration, closed forms,
invariants).  What is not pinned is whether the MI300 kernels the pages
describe use this block layout and zero-point convention: the pages do not
say, so the oracle follows the stated reading, not a printed result.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qro.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Values repeated from qro.h (0..3 follow QuickReduceRegime on the vLLM
# quick_all_reduce API page; 4..6 are fp8 and the asymmetric formats).
F16, BF16, BF16_AS_F16 = 0, 1, 2
FP, Q8, Q6, Q4, FP8, Q8A, Q4A = 0, 1, 2, 3, 4, 5, 6
BLOCK = 32

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, contraction off)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                                  os.path.getmtime(os.path.join(_HERE, "qro.h")))):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _bind(lib):
    u16, u8, f32 = ctypes.c_uint16, ctypes.c_uint8, ctypes.c_float
    sz, i = ctypes.c_size_t, ctypes.c_int
    vp = ctypes.c_void_p
    for name, res, args in [
        ("qro_f16_to_f32", f32, [u16]),
        ("qro_f32_to_f16", u16, [f32]),
        ("qro_f32_to_f16_satfinite", u16, [f32]),
        ("qro_bf16_to_f32", f32, [u16]),
        ("qro_f32_to_bf16", u16, [f32]),
        ("qro_e4m3_to_f32", f32, [u8]),
        ("qro_f32_to_e4m3_satfinite", u8, [f32]),
        ("qro_encoded_bytes", sz, [i, sz]),
        ("qro_quantize", i, [i, i, vp, sz, vp]),
        ("qro_dequantize", i, [i, i, vp, sz, vp]),
        ("qro_allreduce", i, [i, i, i, i, vp, sz, vp, vp]),
    ]:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_u16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype.itemsize != 2:
        raise TypeError("expected 16-bit values (fp16 or bf16 bit patterns)")
    return x.view(np.uint16).reshape(-1)


# ----- scalar conversions (vectorised by looping; small arrays only) -----

def _vec(fn, arr, out_dtype):  # noqa: D103
    return np.array([fn(v) for v in arr.tolist()], dtype=out_dtype)


def f16_to_f32(bits):
    return _vec(_load().qro_f16_to_f32, np.asarray(bits, np.uint16).reshape(-1), np.float32)


def f32_to_f16(v):
    return _vec(_load().qro_f32_to_f16, np.asarray(v, np.float32).reshape(-1), np.uint16)


def f32_to_f16_satfinite(v):
    return _vec(_load().qro_f32_to_f16_satfinite, np.asarray(v, np.float32).reshape(-1), np.uint16)


def bf16_to_f32(bits):
    return _vec(_load().qro_bf16_to_f32, np.asarray(bits, np.uint16).reshape(-1), np.float32)


def f32_to_bf16(v):
    return _vec(_load().qro_f32_to_bf16, np.asarray(v, np.float32).reshape(-1), np.uint16)


def e4m3_to_f32(codes):
    return _vec(_load().qro_e4m3_to_f32, np.asarray(codes, np.uint8).reshape(-1), np.float32)


def f32_to_e4m3_satfinite(v):
    return _vec(_load().qro_f32_to_e4m3_satfinite, np.asarray(v, np.float32).reshape(-1), np.uint8)


# ----- message-level calls -----

def encoded_bytes(fmt: int, n: int) -> int:
    return int(_load().qro_encoded_bytes(fmt, n))


def quantize(dtype: int, fmt: int, x: np.ndarray) -> np.ndarray:
    """Encode n 16-bit values; returns the encoded message as uint8."""
    x = _as_u16(x)
    n = x.size
    enc = np.zeros(max(encoded_bytes(fmt, n), 1), np.uint8)
    if _load().qro_quantize(dtype, fmt, _ptr(x), n, _ptr(enc)) != 0:
        raise ValueError("qro_quantize rejected its arguments")
    return enc[:encoded_bytes(fmt, n)]


def dequantize(dtype: int, fmt: int, enc: np.ndarray, n: int) -> np.ndarray:
    """Decode an encoded message to n 16-bit values (uint16 bit patterns)."""
    enc = np.ascontiguousarray(enc, np.uint8)
    if enc.size < encoded_bytes(fmt, n):
        raise ValueError("encoded buffer too small")
    out = np.zeros(max(n, 1), np.uint16)
    if _load().qro_dequantize(dtype, fmt, _ptr(enc), n, _ptr(out)) != 0:
        raise ValueError("qro_dequantize rejected its arguments")
    return out[:n]


def allreduce(dtype: int, fmt: int, stages: int, inputs, want_wire: bool = True):
    """Emulated allreduce of W equal-length messages.

    Returns (out, wire): out as uint16 bit patterns, wire as uint8 (None for
    stages == 1 or when want_wire is False)."""
    xs = [_as_u16(x) for x in inputs]
    W = len(xs)
    n = xs[0].size if xs else 0
    if any(x.size != n for x in xs):
        raise ValueError("all ranks must hold n elements")
    arr = (ctypes.c_void_p * max(W, 1))(*[x.ctypes.data for x in xs])
    out = np.zeros(max(n, 1), np.uint16)
    wire = None
    wire_ptr = None
    if stages == 2 and want_wire:
        wire = np.zeros(max(encoded_bytes(fmt, n), 1), np.uint8)
        wire_ptr = _ptr(wire)
    rc = _load().qro_allreduce(W, dtype, fmt, stages,
                               ctypes.cast(arr, ctypes.c_void_p), n, _ptr(out), wire_ptr)
    if rc != 0:
        raise ValueError("qro_allreduce rejected its arguments")
    if wire is not None:
        wire = wire[:encoded_bytes(fmt, n)]
    return out[:n], wire


class Oracle:
    """The same API as this module over another build of the oracle source
    (used by the tests that plant mistakes in a copy of qro.c and check that
    the pins catch them)."""

    F16, BF16, BF16_AS_F16 = F16, BF16, BF16_AS_F16
    FP, Q8, Q6, Q4, FP8, Q8A, Q4A = FP, Q8, Q6, Q4, FP8, Q8A, Q4A
    BLOCK = BLOCK

    def __init__(self, so_path: str):
        self._lib = _bind(ctypes.CDLL(so_path))

    def __getattr__(self, name):
        fn = globals().get(name)
        if not callable(fn) or name.startswith("_") or name in ("build", "compile_source"):
            raise AttributeError(name)

        def call(*args, **kwargs):
            global _lib
            saved = _lib
            _lib = self._lib
            try:
                return fn(*args, **kwargs)
            finally:
                _lib = saved
        return call


def compile_source(src_path: str, out_path: str) -> str:
    """Compile a copy of the oracle source with the oracle's flags."""
    subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", out_path, src_path, "-lm"], check=True)
    return out_path
