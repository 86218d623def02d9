"""qr_allreduce_host: the allreduce on host buffers, chunked through a device
workspace with the copies overlapping the kernels.  The method is defined
block by block, so its output and stage-2 payload must equal the oracle's
bit for bit for any chunk size: one chunk, many chunks, a ragged last chunk,
page-locked and pageable host memory."""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import BF16, F16, FP, FP8, Q4, Q4A, Q6, Q8, Q8A, to_bits

BF16_AS_F16 = qr.BF16_AS_F16

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
    src = BF16 if dtype == BF16_AS_F16 else dtype
    return [to_bits((rng.standard_normal(n) * np.exp2(rng.uniform(-3, 3))).astype(np.float32), src)
            for _ in range(W)]


def host_buffer(nbytes, pinned):
    t = torch.empty(nbytes, dtype=torch.uint8)
    return t.pin_memory() if pinned else t


def run_host(W, dtype, fmt, stages, xs, chunk, pinned, want_wire=True):
    n = xs[0].size
    ins = []
    for x in xs:
        t = host_buffer(2 * n, pinned)
        t.numpy()[:] = np.ascontiguousarray(x).view(np.uint8)
        ins.append(t)
    out = host_buffer(2 * n + 64, pinned)
    out.numpy()[:] = 0xA5
    wire = None
    wbytes = qr.qr_encoded_bytes(fmt, n)
    if stages == 2 and want_wire:
        wire = host_buffer(wbytes + 64, pinned)
        wire.numpy()[:] = 0xA5
    ws = qr.host_workspace(W, fmt, chunk)
    qr.qr_allreduce_host(W, dtype, fmt, stages, ins, n, out, wire, ws, chunk_elems=chunk)
    torch.cuda.current_stream().synchronize()
    assert (out.numpy()[2 * n:] == 0xA5).all(), "write past the output"
    if wire is not None:
        assert (wire.numpy()[wbytes:] == 0xA5).all(), "write past the payload"
    return out.numpy()[:2 * n].view(np.uint16), (wire.numpy()[:wbytes] if wire is not None else None)


@pytest.mark.parametrize("W,dtype,fmt,stages,n,chunk,pinned", [
    (2, F16, Q8, 2, 1 << 20, 1 << 17, True),             # 8 chunks
    (2, F16, Q4, 2, (1 << 20) + 8200, 1 << 18, True),    # ragged last chunk, ragged last block
    (4, BF16, Q4A, 2, 300000, 65536, True),
    (8, F16, FP8, 2, 123456, 32768, True),
    (2, BF16, Q6, 2, 40000, 1 << 21, True),              # one chunk larger than the message
    (2, F16, FP, 2, 500000, 1 << 16, True),
    (4, F16, Q8A, 1, 262144 + 40, 1 << 15, True),        # one stage
    (2, BF16_AS_F16, Q8, 2, 200000, 1 << 15, True),      # bf16 -> fp16 cast option
    (2, F16, Q8, 2, 300000, 1 << 16, False),             # pageable host memory
    (1, F16, Q4, 2, 70000, 8192, True),                  # W = 1
    (2, F16, Q8, 2, 5 * (1 << 22) + 96, 1 << 22, True),  # chunks on the pipeline kernel
])
def test_host_entry_matches_oracle(oracle_mod, W, dtype, fmt, stages, n, chunk, pinned):
    xs = messages(8000 + W * 10 + fmt, W, n, dtype)
    out, wire = run_host(W, dtype, fmt, stages, xs, chunk, pinned)
    o_out, o_wire = oracle_mod.allreduce(dtype, fmt, stages, xs)
    bad = np.nonzero(out != o_out)[0]
    assert bad.size == 0, f"{bad.size} output elements differ, first at {bad[:5]}"
    if stages == 2:
        assert np.array_equal(wire, o_wire), "stage-2 payload differs"


def test_host_entry_without_payload_and_back_to_back(oracle_mod):
    W, dtype, fmt, n, chunk = 2, F16, Q6, 250000, 1 << 15
    for call in range(3):  # consecutive calls reuse the library's copy streams and events
        xs = messages(8100 + call, W, n, dtype)
        out, _ = run_host(W, dtype, fmt, 2, xs, chunk, True, want_wire=False)
        o_out, _ = oracle_mod.allreduce(dtype, fmt, 2, xs, want_wire=False)
        assert np.array_equal(out, o_out), f"output differs on call {call + 1}"


def test_host_entry_on_a_side_stream_orders_with_that_stream(oracle_mod):
    W, dtype, fmt, n, chunk = 4, BF16, Q8, 400000, 1 << 16
    xs = messages(8200, W, n, dtype)
    ins = [torch.from_numpy(x.view(np.int16).copy()).pin_memory() for x in xs]
    out = torch.empty(n, dtype=torch.int16).pin_memory()
    ws = qr.host_workspace(W, fmt, chunk)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        ws.zero_()  # work already on the stream: the call must come after it
        qr.qr_allreduce_host(W, dtype, fmt, 1, ins, n, out, None, ws, chunk_elems=chunk)
    side.synchronize()
    o_out, _ = oracle_mod.allreduce(dtype, fmt, 1, xs)
    assert np.array_equal(out.numpy().view(np.uint16), o_out)
