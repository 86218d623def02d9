"""The kernel-path table decides which kernel serves a call: a message of
exactly the selected limit runs the direct kernel and one 8-element step past
it the pipeline kernel (seen as the kernel node of a captured CUDA graph), for
shapes of every mode; the override reroutes every shape and restoring the
table undoes it."""
import numpy as np
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
    names = sorted(set(re.findall(r"qr_(?:direct|encode|pipeline|decode)_kernel", text)))
    assert names, "no qr kernel node in the captured graph"
    return names


def path_of(names):
    """The path a call took: the direct kernel (qr_encode_kernel for
    encode-only calls) or the pipeline kernel."""
    direct = any("qr_direct_kernel" in nm or "qr_encode_kernel" in nm for nm in names)
    pipe = any("qr_pipeline_kernel" in nm for nm in names)
    assert direct != pipe, names
    return "direct" if direct else "pipeline"


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
def test_routing_follows_the_table(bufs, W, dtype, fmt, stages):
    assert qr.qr_direct_limit() == qr.DIRECT_LIMIT_TABLE
    limit = qr.qr_selected_direct_limit(W, dtype, fmt, stages)
    probes = []
    if limit > 0:
        n = min(limit, MAX_TEST_N) // 8 * 8
        probes.append((n, "direct"))
    if limit < MAX_TEST_N:
        probes.append((limit + 8 if limit else 8192, "pipeline"))
    for n, want in probes:
        assert path_of(kernels_launched(run(W, dtype, fmt, stages, n, bufs))) == want, (n, limit)


def test_override_reroutes_every_shape_and_the_table_comes_back(bufs):
    W, dtype, fmt, stages = 2, F16, Q8, 2
    limit = qr.qr_selected_direct_limit(W, dtype, fmt, stages)
    try:
        qr.qr_set_direct_limit(0)
        assert path_of(kernels_launched(run(W, dtype, fmt, stages, 4096, bufs))) == "pipeline"
        qr.qr_set_direct_limit(qr.MAX_ELEMS)
        assert path_of(kernels_launched(run(W, dtype, fmt, stages, 1 << 22, bufs))) == "direct"
    finally:
        qr.qr_set_direct_limit(qr.DIRECT_LIMIT_TABLE)
    assert qr.qr_selected_direct_limit(W, dtype, fmt, stages) == limit
    np.testing.assert_equal(qr.qr_direct_limit(), qr.DIRECT_LIMIT_TABLE)
