"""The kernel-path tables decide which kernel serves a call: a message of
exactly the direct limit runs the direct kernel, one 8-element step past it
the narrow-tile pipeline where the shape has a narrow-tile range, and one
step past the narrow-tile limit the wide-tile pipeline (seen as the kernel
node of a captured CUDA graph, the pipeline's tile width being its last
template argument), for shapes of every mode; a forced path reroutes every
shape and restoring the tables undoes it."""
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import BF16, F16, FP, FP8, Q4, Q4A, Q6, Q8, Q8A

pytestmark = pytest.mark.gpu

MAX_TEST_N = 64 << 20  # largest message the test routes (elements per rank)


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qr.lib()
    qr.qr_device_error(clear=True)
    yield
    assert qr.qr_device_error(clear=True) == 0


def _dot_print(g, path):
    """Write the DOT description of the captured graph g to path: torch's
    debug_dump, else cudaGraphDebugDotPrint from the process's libcudart on
    the raw graph handle."""
    import ctypes
    import os
    g.debug_dump(path)
    if os.path.exists(path):
        return
    libs = [ln.split()[-1] for ln in open("/proc/self/maps") if "libcudart.so" in ln]
    assert libs, "no libcudart loaded"
    cudart = ctypes.CDLL(libs[0])
    cudart.cudaGraphDebugDotPrint.argtypes = [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint]
    cudart.cudaGraphDebugDotPrint.restype = ctypes.c_int
    assert cudart.cudaGraphDebugDotPrint(ctypes.c_void_p(g.raw_cuda_graph()), path.encode(), 1) == 0
    assert os.path.exists(path)


def kernels_launched(fn):
    """Names of the kernels fn launches, read from the DOT description of a
    CUDA graph that captures fn (each launch is a kernel node labelled with
    the kernel's name)."""
    import os
    import re
    import tempfile
    fn()  # first-call set-up outside the capture
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)  # keep the cudaGraph_t after capture
    except TypeError:
        g = torch.cuda.CUDAGraph()
    g.enable_debug_mode()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize()
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "graph.dot")
        _dot_print(g, path)
        text = open(path).read()
    del g
    names = set()
    # demangled "qr_pipeline_kernel<3, 0, 2, 2, 4>" or mangled "qr_pipeline_kernelILi3ELi0E...E"
    for m in re.finditer(r"qr_(direct|block|encode|pipeline|decode)_kernel(<[^>]*>|I(?:Li-?\d+E)+E)?", text):
        names.add((m.group(1), tuple(int(v) for v in re.findall(r"-?\d+", m.group(2) or ""))))
    assert names, "no qr kernel node in the captured graph"
    return sorted(names)


def path_of(names):
    """The path a call took: PATH_DIRECT (qr_direct_kernel; qr_block_kernel for
    the larger W=2 and W=4 calls of the integer formats; qr_encode_kernel for
    encode-only calls), else the pipeline with narrow or wide tiles (the
    pipeline kernel's fifth template argument: consumer warps per tile)."""
    kinds = {k for k, _ in names}
    assert len(kinds) == 1, names
    kind = kinds.pop()
    if kind in ("direct", "block", "encode"):
        return qr.PATH_DIRECT
    assert kind == "pipeline", names
    widths = {a[4] for _, a in names if len(a) == 5}
    assert len(widths) == 1, names
    return qr.PATH_PIPELINE_NARROW if widths.pop() == 4 else qr.PATH_PIPELINE


def run(W, dtype, fmt, stages, n, bufs):
    ins, out, wire = bufs
    if stages == 0:
        return lambda: qr.qr_quantize(dtype, fmt, ins[0], n, wire)
    return lambda: qr.qr_allreduce_emulated(W, dtype, fmt, stages, ins[:W], n, out, wire if stages == 2 else None)


@pytest.fixture(scope="module")
def bufs():
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    ins = [torch.randn(MAX_TEST_N + 64, device="cuda", generator=g).half().view(torch.int16) for _ in range(8)]
    out = torch.empty(MAX_TEST_N + 64, dtype=torch.int16, device="cuda")
    wire = torch.empty(2 * (MAX_TEST_N + 64), dtype=torch.uint8, device="cuda")
    return ins, out, wire


SHAPES = [(1, F16, Q4, 0), (1, BF16, Q8A, 0), (2, F16, Q8, 2), (2, F16, FP, 1), (4, BF16, Q4A, 2),
          (4, F16, Q6, 1), (8, F16, FP8, 2), (8, BF16, Q8, 1), (8, 2, Q4, 2), (2, 2, FP, 2)]


@pytest.mark.parametrize("W,dtype,fmt,stages", SHAPES)
def test_routing_follows_the_tables(bufs, W, dtype, fmt, stages):
    from select_table_util import expected_path, limits, parse_tables
    assert qr.qr_forced_kernel_path() == qr.PATH_TABLE
    tabs = parse_tables()
    l1, l2 = limits(tabs, W, dtype, fmt, stages)
    probes = sorted({n for n in (8, l1, l1 + 8, l2, l2 + 8) if 8 <= n <= MAX_TEST_N})
    for n in probes:
        want = expected_path(tabs, W, dtype, fmt, stages, n)
        assert qr.qr_kernel_path(W, dtype, fmt, stages, n) == want
        if want == qr.PATH_PIPELINE_NARROW and W == 8:
            want = qr.PATH_PIPELINE  # narrow tiles are built for W <= 4 only
        assert path_of(kernels_launched(run(W, dtype, fmt, stages, n, bufs))) == want, (n, l1, l2)


def test_forced_path_reroutes_every_shape_and_the_tables_come_back(bufs):
    W, dtype, fmt, stages = 2, F16, Q8, 2
    sizes = (4096, 1 << 22, 1 << 25)
    before = [qr.qr_kernel_path(W, dtype, fmt, stages, n) for n in sizes]
    for path, n in ((qr.PATH_PIPELINE, 4096), (qr.PATH_PIPELINE_NARROW, 4096), (qr.PATH_DIRECT, 1 << 22)):
        with qr.forced_kernel_path(path):
            assert qr.qr_kernel_path(W, dtype, fmt, stages, n) == path
            assert path_of(kernels_launched(run(W, dtype, fmt, stages, n, bufs))) == path
    assert qr.qr_forced_kernel_path() == qr.PATH_TABLE
    assert [qr.qr_kernel_path(W, dtype, fmt, stages, n) for n in sizes] == before
