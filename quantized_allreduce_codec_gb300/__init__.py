"""GB300 quick-allreduce codec: thin Python binding of libqr.so (include/qr.h).

Argument marshalling only: every step of the data path runs in the CUDA
kernels of libqr.so.  If the library has not been built this module raises
on first use; there is no fallback.  Build with
``python -m quantized_allreduce_codec_gb300.build``.

Functions take torch tensors (device memory, contiguous) or raw integer
device addresses; ``stream`` defaults to torch's current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

F16, BF16, BF16_AS_F16 = 0, 1, 2
QR_FP, QR_Q8, QR_Q6, QR_Q4, QR_FP8, QR_Q8_ASYM, QR_Q4_ASYM = 0, 1, 2, 3, 4, 5, 6
FORMATS = {"FP": QR_FP, "Q8": QR_Q8, "Q6": QR_Q6, "Q4": QR_Q4, "FP8": QR_FP8,
           "Q8A": QR_Q8_ASYM, "Q4A": QR_Q4_ASYM}
STATUS = ["QR_OK", "QR_ERR_NULL", "QR_ERR_DTYPE", "QR_ERR_FORMAT", "QR_ERR_WORLD",
          "QR_ERR_STAGES", "QR_ERR_SIZE", "QR_ERR_ALIGN", "QR_ERR_OVERLAP", "QR_ERR_CUDA",
          "QR_ERR_DEVICE", "QR_ERR_SCRATCH", "QR_ERR_PATH"]
# kernel paths (qr_path)
PATH_TABLE, PATH_DIRECT, PATH_PIPELINE_NARROW, PATH_PIPELINE = -1, 0, 1, 2
PATH_NAMES = {PATH_DIRECT: "direct", PATH_PIPELINE_NARROW: "pipeline_narrow", PATH_PIPELINE: "pipeline"}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqr.so")
EXPORTS = ("qr_encoded_bytes", "qr_quantize", "qr_dequantize", "qr_allreduce_emulated",
           "qr_status_string", "qr_device_error", "qr_kernel_path", "qr_set_kernel_path",
           "qr_forced_kernel_path", "qr_selftest_wait_timeout", "qr_selftest_reciprocal", "qr_stage1_bytes", "qr_allreduce_staged",
           "qr_allreduce_staged_noalloc", "qr_host_workspace_bytes", "qr_allreduce_host")
MAX_ELEMS = 1 << 36  # QR_MAX_ELEMS: the largest message (elements)
DEFAULT_HOST_CHUNK = 1 << 22  # elements per rank per chunk of qr_allreduce_host (8 MiB of fp16)

_lib = None
_lock = threading.Lock()


class QRError(RuntimeError):
    """A libqr call returned a status other than QR_OK."""

    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS[status] if 0 <= status < len(STATUS) else str(status)
        super().__init__(f"{what}: {name} ({qr_status_string(status)})")


def lib():
    """The loaded libqr.so (ctypes.CDLL); raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"libqr.so not built ({LIB_PATH}); run "
                                       "python -m quantized_allreduce_codec_gb300.build")
                L = ctypes.CDLL(LIB_PATH)
                vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
                L.qr_encoded_bytes.restype = sz
                L.qr_encoded_bytes.argtypes = [i, sz]
                L.qr_quantize.restype = i
                L.qr_quantize.argtypes = [i, i, vp, sz, vp, vp]
                L.qr_dequantize.restype = i
                L.qr_dequantize.argtypes = [i, i, vp, sz, vp, vp]
                L.qr_allreduce_emulated.restype = i
                L.qr_allreduce_emulated.argtypes = [i, i, i, i, vp, sz, vp, vp, vp]
                L.qr_status_string.restype = ctypes.c_char_p
                L.qr_status_string.argtypes = [i]
                L.qr_device_error.restype = i
                L.qr_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
                L.qr_kernel_path.restype = i
                L.qr_kernel_path.argtypes = [i, i, i, i, sz]
                L.qr_set_kernel_path.restype = i
                L.qr_set_kernel_path.argtypes = [i]
                L.qr_forced_kernel_path.restype = i
                L.qr_forced_kernel_path.argtypes = []
                L.qr_stage1_bytes.restype = sz
                L.qr_stage1_bytes.argtypes = [i, i, sz]
                L.qr_allreduce_staged.restype = i
                L.qr_allreduce_staged.argtypes = [i, i, i, vp, sz, vp, vp, vp, vp]
                L.qr_allreduce_staged_noalloc.restype = i
                L.qr_allreduce_staged_noalloc.argtypes = [i, i, i, vp, sz, vp, vp, vp]
                L.qr_host_workspace_bytes.restype = sz
                L.qr_host_workspace_bytes.argtypes = [i, i, sz]
                L.qr_allreduce_host.restype = i
                L.qr_allreduce_host.argtypes = [i, i, i, i, vp, sz, vp, vp, vp, sz, sz, vp]
                L.qr_selftest_wait_timeout.restype = i
                L.qr_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
                L.qr_selftest_reciprocal.restype = i
                L.qr_selftest_reciprocal.argtypes = [vp, vp]
                _lib = L
    return _lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "__array_interface__"):  # numpy array (host memory)
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("arrays must be C-contiguous")
        return x.ctypes.data
    if not x.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _check(st: int, what: str):
    if st != 0:
        raise QRError(st, what)


def _dtype_code(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    import torch
    if dtype == torch.float16:
        return F16
    if dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported dtype {dtype}")


def _rank_pointers(inputs, W: int, what: str):
    """Host array of the W rank pointers, as the C calls read it.  The C side
    reads exactly W entries, so a list of any other length is refused here
    instead of being read past its end."""
    if len(inputs) != W:
        raise ValueError(f"{what}: {len(inputs)} rank buffers given for W={W}")
    if not inputs:
        return None
    ptrs = (ctypes.c_void_p * len(inputs))(*[_addr(x) for x in inputs])
    return ctypes.cast(ptrs, ctypes.c_void_p)


def qr_status_string(status: int) -> str:
    return lib().qr_status_string(status).decode()


def qr_encoded_bytes(fmt: int, n: int) -> int:
    return int(lib().qr_encoded_bytes(fmt, n))


def qr_quantize(dtype, fmt: int, inp, n: int, enc, stream=None) -> None:
    """Encode n values of `inp` into `enc` (qr_encoded_bytes(fmt, n) bytes)."""
    _check(lib().qr_quantize(_dtype_code(dtype), fmt, _addr(inp), n, _addr(enc), _stream(stream)),
           "qr_quantize")


def qr_dequantize(dtype, fmt: int, enc, n: int, out, stream=None) -> None:
    """Decode an encoded message into n values of `out`."""
    _check(lib().qr_dequantize(_dtype_code(dtype), fmt, _addr(enc), n, _addr(out), _stream(stream)),
           "qr_dequantize")


def qr_allreduce_emulated(W: int, dtype, fmt: int, stages: int, inputs, n: int, out,
                          wire=None, stream=None) -> None:
    """Emulated allreduce of W rank messages (list of W tensors / addresses)."""
    ptrs = _rank_pointers(inputs, W, "qr_allreduce_emulated")
    _check(lib().qr_allreduce_emulated(W, _dtype_code(dtype), fmt, stages, ptrs, n,
                                       _addr(out), _addr(wire), _stream(stream)),
           "qr_allreduce_emulated")


def qr_device_error(clear: bool = True) -> int:
    """Synchronise and return the kernels' wait-limit flags (0 = none)."""
    flags = ctypes.c_uint(0)
    st = lib().qr_device_error(ctypes.byref(flags), 1 if clear else 0)
    if st not in (0, 10):
        raise QRError(st, "qr_device_error")
    return int(flags.value)


def qr_kernel_path(W: int, dtype, fmt: int, stages: int, n: int) -> int:
    """The kernel a call of this shape and size runs now (PATH_DIRECT,
    PATH_PIPELINE_NARROW or PATH_PIPELINE; stages 0: qr_quantize); -1 for a
    shape no call can have."""
    return int(lib().qr_kernel_path(W, _dtype_code(dtype), fmt, stages, n))


def qr_set_kernel_path(path: int) -> None:
    """Force one kernel path for every call in the process (PATH_TABLE
    restores the measured tables).  Process-global: other threads are
    rerouted too."""
    _check(lib().qr_set_kernel_path(path), "qr_set_kernel_path")


def qr_forced_kernel_path() -> int:
    """The forced kernel path, or PATH_TABLE when the measured tables route."""
    return int(lib().qr_forced_kernel_path())


class forced_kernel_path:
    """Context manager: force `path` for the calls inside, then restore the
    previous setting (process-global, like qr_set_kernel_path)."""

    def __init__(self, path: int):
        self.path = path

    def __enter__(self):
        self.old = qr_forced_kernel_path()
        qr_set_kernel_path(self.path)
        return self

    def __exit__(self, *exc):
        qr_set_kernel_path(self.old)
        return False


def qr_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self-test (raises device flag 8 after limit_us)."""
    _check(lib().qr_selftest_wait_timeout(limit_us, _stream(stream)), "qr_selftest_wait_timeout")


SELFTEST_RECIPROCALS = 0x7BFF


def qr_selftest_reciprocal(out, stream=None) -> None:
    """The direct kernel's block-scale reciprocal of every positive finite
    fp16 value (bit patterns 1 .. 0x7BFF) into the float32 device tensor out
    (at least SELFTEST_RECIPROCALS elements)."""
    if out.numel() * out.element_size() < 4 * SELFTEST_RECIPROCALS:
        raise ValueError("out holds fewer than SELFTEST_RECIPROCALS floats")
    _check(lib().qr_selftest_reciprocal(_addr(out), _stream(stream)), "qr_selftest_reciprocal")

def qr_stage1_bytes(W: int, fmt: int, n: int) -> int:
    """Bytes of the stage-1 exchange buffer of qr_allreduce_staged."""
    return int(lib().qr_stage1_bytes(W, fmt, n))


def qr_allreduce_staged(W: int, dtype, fmt: int, inputs, n: int, out, wire, stage1,
                        stream=None) -> None:
    """Two-stage allreduce with the stage-1 exchange materialised in `stage1`."""
    ptrs = _rank_pointers(inputs, W, "qr_allreduce_staged")
    _check(lib().qr_allreduce_staged(W, _dtype_code(dtype), fmt, ptrs, n,
                                     _addr(out), _addr(wire), _addr(stage1), _stream(stream)),
           "qr_allreduce_staged")


NOALLOC_SCRATCH_BYTES = 16 << 20


def qr_allreduce_staged_noalloc(W: int, dtype, fmt: int, inputs, n: int, out, wire,
                                stream=None) -> None:
    """qr_allreduce_staged with the library's built-in stage-1 array instead
    of a caller buffer, for callers that cannot allocate device memory (for
    example while a CUDA graph is being captured).  Messages needing more
    than NOALLOC_SCRATCH_BYTES of stage-1 space raise QR_ERR_SCRATCH; calls
    that overlap on the GPU share the array and race."""
    ptrs = _rank_pointers(inputs, W, "qr_allreduce_staged_noalloc")
    _check(lib().qr_allreduce_staged_noalloc(W, _dtype_code(dtype), fmt, ptrs, n,
                                             _addr(out), _addr(wire), _stream(stream)),
           "qr_allreduce_staged_noalloc")


def qr_host_workspace_bytes(W: int, fmt: int, chunk_elems: int = DEFAULT_HOST_CHUNK) -> int:
    """Device workspace bytes qr_allreduce_host needs (0: invalid arguments)."""
    return int(lib().qr_host_workspace_bytes(W, fmt, chunk_elems))


def host_workspace(W: int, fmt: int, chunk_elems: int = DEFAULT_HOST_CHUNK, device=None):
    """A device byte tensor large enough to serve as qr_allreduce_host's
    workspace (memory from torch's allocator)."""
    import torch
    nbytes = qr_host_workspace_bytes(W, fmt, chunk_elems)
    if nbytes == 0:
        raise ValueError("invalid W, format or chunk size")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def qr_allreduce_host(W: int, dtype, fmt: int, stages: int, host_inputs, n: int, host_out,
                      host_wire=None, workspace=None, workspace_bytes: int | None = None,
                      chunk_elems: int = DEFAULT_HOST_CHUNK, stream=None) -> None:
    """qr_allreduce_emulated on host buffers (CPU tensors or numpy arrays,
    page-locked for overlapped copies), chunked through a device workspace
    (see host_workspace); the copies and the kernels overlap."""
    if workspace is None:
        raise ValueError("qr_allreduce_host needs a device workspace (see host_workspace)")
    if workspace_bytes is None:
        if isinstance(workspace, int):
            raise ValueError("workspace_bytes is required with a raw workspace address")
        workspace_bytes = workspace.numel() * workspace.element_size()
    ptrs = _rank_pointers(host_inputs, W, "qr_allreduce_host")
    _check(lib().qr_allreduce_host(W, _dtype_code(dtype), fmt, stages, ptrs, n,
                                   _addr(host_out), _addr(host_wire), _addr(workspace), workspace_bytes,
                                   chunk_elems, _stream(stream)),
           "qr_allreduce_host")
