"""Every entry point is stream-ordered and allocates nothing on the device
during a call, so a sequence of calls can be captured into a CUDA graph once
and replayed.  A replay after new values were copied into the captured input
buffers must give the oracle's bits for those values, replay after replay
(output and stage-2 payload)."""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import BF16, F16, FP, FP8, Q4, Q4A, Q6, Q8, Q8A, to_bits

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
    return [to_bits((rng.standard_normal(n) * np.exp2(rng.uniform(-3, 3))).astype(np.float32), dtype)
            for _ in range(W)]


def load(dev, host_bits):
    dev.copy_(torch.from_numpy(np.ascontiguousarray(host_bits).view(np.int16)))


def capture(fn):
    """Warm up fn on a side stream (first-use set-up happens outside the
    capture), then capture it into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def host_bits(t, n):
    return t[:n].cpu().numpy().view(np.uint16)


# n spans the direct kernel (small) and the pipeline kernel (above the
# default 4M-element limit), with ragged tails
@pytest.mark.parametrize("W,dtype,fmt,stages,n", [
    (2, F16, Q8, 2, 5 * 8192 + 96),
    (4, BF16, Q4A, 2, 64 * 1024 + 40),
    (8, F16, FP8, 1, 3 * 8192),
    (2, BF16, Q6, 2, (1 << 22) + 8192 + 8),
    (2, F16, FP, 2, (1 << 22) + 1024),
    (4, F16, Q8A, 1, (1 << 22) + 32),
])
def test_allreduce_graph_replays_match_oracle(oracle_mod, W, dtype, fmt, stages, n):
    ins = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(W)]
    out = torch.zeros(n, dtype=torch.int16, device="cuda")
    # one stage has no stage-2 payload: the call takes no wire buffer then
    wire = torch.zeros(qr.qr_encoded_bytes(fmt, n), dtype=torch.uint8, device="cuda") if stages == 2 else None
    g = capture(lambda: qr.qr_allreduce_emulated(W, dtype, fmt, stages, ins, n, out, wire))
    for rep in range(2):
        xs = messages(7000 + 13 * rep + fmt, W, n, dtype)
        for t, x in zip(ins, xs):
            load(t, x)
        g.replay()
        torch.cuda.synchronize()
        o_out, o_wire = oracle_mod.allreduce(dtype, fmt, stages, xs)
        assert np.array_equal(host_bits(out, n), o_out), f"output differs on replay {rep}"
        if stages == 2:
            assert np.array_equal(wire.cpu().numpy(), o_wire), f"payload differs on replay {rep}"


@pytest.mark.parametrize("dtype,fmt,n", [(F16, Q4, 8192 * 7 + 64), (BF16, Q8A, (1 << 22) + 4096)])
def test_codec_round_trip_graph_replays_match_oracle(oracle_mod, dtype, fmt, n):
    x = torch.zeros(n, dtype=torch.int16, device="cuda")
    enc = torch.zeros(qr.qr_encoded_bytes(fmt, n), dtype=torch.uint8, device="cuda")
    y = torch.zeros(n, dtype=torch.int16, device="cuda")

    def step():
        qr.qr_quantize(dtype, fmt, x, n, enc)
        qr.qr_dequantize(dtype, fmt, enc, n, y)

    g = capture(step)
    for rep in range(2):
        xb = messages(7100 + rep, 1, n, dtype)[0]
        load(x, xb)
        g.replay()
        torch.cuda.synchronize()
        o_enc = oracle_mod.quantize(dtype, fmt, xb)
        assert np.array_equal(enc.cpu().numpy(), o_enc), f"encoding differs on replay {rep}"
        assert np.array_equal(host_bits(y, n), oracle_mod.dequantize(dtype, fmt, o_enc, n))


def test_staged_without_allocation_graph_replays_match_oracle(oracle_mod):
    W, dtype, fmt, n = 4, F16, Q6, 6 * 8192 + 24
    assert qr.qr_stage1_bytes(W, fmt, n) <= qr.NOALLOC_SCRATCH_BYTES
    ins = [torch.zeros(n, dtype=torch.int16, device="cuda") for _ in range(W)]
    out = torch.zeros(n, dtype=torch.int16, device="cuda")
    wire = torch.zeros(qr.qr_encoded_bytes(fmt, n), dtype=torch.uint8, device="cuda")
    g = capture(lambda: qr.qr_allreduce_staged_noalloc(W, dtype, fmt, ins, n, out, wire))
    for rep in range(2):
        xs = messages(7200 + rep, W, n, dtype)
        for t, x in zip(ins, xs):
            load(t, x)
        g.replay()
        torch.cuda.synchronize()
        o_out, o_wire = oracle_mod.allreduce(dtype, fmt, 2, xs)
        assert np.array_equal(host_bits(out, n), o_out), f"output differs on replay {rep}"
        assert np.array_equal(wire.cpu().numpy(), o_wire), f"payload differs on replay {rep}"
