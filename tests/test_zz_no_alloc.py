"""qr_allreduce_staged_noalloc, the staged allreduce for callers that cannot
allocate device memory (code running under CUDA-graph capture, plugins that
are only handed input and output pointers, paths where cudaMalloc/cudaFree
are not allowed): it uses a fixed stage-1 array inside the library instead of
a caller buffer.  Its results must equal qr_allreduce_staged's (the entry
point that takes the buffer from the caller) bit for bit, also on the second
of two calls in a row, which finds the first call's bytes in the shared
array.  This file runs last in the suite and also passes on its own."""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import BF16, F16, FP, FP8, Q4A, Q6, Q8, to_bits
from qr_gpu_util import dev_u16, guard_intact, out_buffer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qr.lib()
    qr.qr_device_error(clear=True)
    yield
    assert qr.qr_device_error(clear=True) == 0


def messages(seed, W, n, dtype):
    rng = np.random.default_rng(seed)
    return [to_bits((rng.standard_normal(n) * np.exp2(rng.uniform(-4, 4))).astype(np.float32), dtype)
            for _ in range(W)]


def with_caller_buffer(W, dtype, fmt, ins, n):
    out, wire = out_buffer(2 * n), out_buffer(qr.qr_encoded_bytes(fmt, n))
    st1 = torch.empty(qr.qr_stage1_bytes(W, fmt, n), dtype=torch.uint8, device="cuda")
    qr.qr_allreduce_staged(W, dtype, fmt, ins, n, out, wire, st1)
    torch.cuda.synchronize()
    return out, wire


def without_allocation(W, dtype, fmt, ins, n):
    wbytes = qr.qr_encoded_bytes(fmt, n)
    out, wire = out_buffer(2 * n), out_buffer(wbytes)
    qr.qr_allreduce_staged_noalloc(W, dtype, fmt, ins, n, out, wire)
    torch.cuda.synchronize()
    assert guard_intact(out, 2 * n) and guard_intact(wire, wbytes)
    return out, wire


@pytest.mark.parametrize("W,dtype,fmt,n", [
    (2, F16, Q8, 64 * 4096),
    (4, BF16, Q4A, 5 * 8192 + 40),
    (8, F16, FP8, 32 * 1000 + 8),
    (8, BF16, Q6, 8 * 8192),
    (2, F16, FP, 65536),
])
def test_noalloc_equals_caller_buffer_on_two_calls_in_a_row(W, dtype, fmt, n):
    assert qr.qr_stage1_bytes(W, fmt, n) <= qr.NOALLOC_SCRATCH_BYTES
    for call in range(2):  # the second call finds the first call's bytes in the array
        ins = [dev_u16(x) for x in messages(9000 + 31 * call + fmt, W, n, dtype)]
        ref_out, ref_wire = with_caller_buffer(W, dtype, fmt, ins, n)
        out, wire = without_allocation(W, dtype, fmt, ins, n)
        assert torch.equal(out[:2 * n], ref_out[:2 * n]), f"output differs on call {call + 1}"
        wb = qr.qr_encoded_bytes(fmt, n)
        assert torch.equal(wire[:wb], ref_wire[:wb]), f"payload differs on call {call + 1}"


def test_noalloc_rejects_messages_beyond_the_array():
    x = torch.zeros(64, dtype=torch.float16, device="cuda")
    n = 8 << 20  # W=2 Q8 needs about 17.8 MB of stage-1 space here
    assert qr.qr_stage1_bytes(2, Q8, n) > qr.NOALLOC_SCRATCH_BYTES
    with pytest.raises(qr.QRError, match="QR_ERR_SCRATCH"):
        qr.qr_allreduce_staged_noalloc(2, F16, Q8, [x, x], n, x, x)
