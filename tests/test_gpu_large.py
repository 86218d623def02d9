"""Messages past 2^31 elements per rank (byte offsets past 2^32): every
index in the kernels is 64-bit, and these checks would catch one that is
not.  The two-stage allreduce (pipeline kernel, then the direct kernel on
the same inputs) is compared with the oracle on sampled blocks, including
the blocks around element 2^31 and the ragged last block; the two kernels
must agree on every element, and decoding the stage-2 payload must give
the output bit for bit, also for the whole message."""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build
from quantized_allreduce_codec_gb300.inputs import F16, Q4, Q8A, long_message_bits
from qr_gpu_util import gather_blocks, split_encoded

pytestmark = pytest.mark.gpu

N_BIG = (1 << 31) + 3 * (1 << 20) + 8  # 4 GiB + 6 MiB + 16 bytes per rank


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qr.lib()
    qr.qr_device_error(clear=True)
    yield
    assert qr.qr_device_error(clear=True) == 0


def boundary_blocks(n, seed):
    nb = (n + 31) // 32
    edge = (1 << 31) // 32  # the block that starts at element 2^31
    picks = {0, 1, nb - 2, nb - 1, edge - 2, edge - 1, edge, edge + 1, (1 << 26) + 8191}
    picks.update(np.random.default_rng(seed).integers(0, nb, 96).tolist())
    return np.array(sorted(p for p in picks if 0 <= p < nb), np.int64)


def device_blocks(t16, blocks, n):
    """The given blocks of a device int16 tensor, concatenated, as uint16."""
    idx = torch.cat([torch.arange(32 * b, min(32 * b + 32, n), device=t16.device) for b in blocks.tolist()])
    return t16[idx].cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", [Q4, Q8A])
def test_two_stage_beyond_2_31_elements(oracle_mod, fmt):
    n, W = N_BIG, 2
    free, _ = torch.cuda.mem_get_info()
    assert free > 30 << 30, "needs about 26 GiB of device memory"
    xs = [long_message_bits(9100 + r + 10 * fmt, n, F16) for r in range(W)]
    ins = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs]
    out = torch.empty(n, dtype=torch.int16, device="cuda")
    wbytes = qr.qr_encoded_bytes(fmt, n)
    wire = torch.empty(wbytes, dtype=torch.uint8, device="cuda")
    with qr.forced_kernel_path(qr.PATH_PIPELINE):
        qr.qr_allreduce_emulated(W, F16, fmt, 2, ins, n, out, wire)

    blocks = boundary_blocks(n, 9200 + fmt)
    sub = [gather_blocks(x, blocks) for x in xs]
    o_out, o_wire = oracle_mod.allreduce(F16, fmt, 2, sub)
    got = device_blocks(out, blocks, n)
    assert np.array_equal(got, o_out), f"{int((got != o_out).sum())} sampled elements differ"
    # the payload of the sampled blocks, region by region
    g_codes, g_scales, g_zps = split_encoded(wire.cpu().numpy(), fmt, n)
    o_codes, o_scales, o_zps = split_encoded(o_wire, fmt, sub[0].size)
    assert np.array_equal(g_codes[blocks], o_codes)
    assert np.array_equal(g_scales[blocks], o_scales)
    if o_zps is not None:
        assert np.array_equal(g_zps[blocks], o_zps)

    # the whole payload decodes to the whole output
    dec = torch.empty_like(out)
    qr.qr_dequantize(F16, fmt, wire, n, dec)
    torch.cuda.synchronize()
    assert torch.equal(dec, out), "decoded payload differs from the output"
    del dec

    # the direct path on the same inputs (at this size the block kernel, one
    # thread per block): the same output and payload
    out2 = torch.empty_like(out)
    wire2 = torch.empty_like(wire)
    with qr.forced_kernel_path(qr.PATH_DIRECT):
        qr.qr_allreduce_emulated(W, F16, fmt, 2, ins, n, out2, wire2)
        torch.cuda.synchronize()
    assert torch.equal(out2, out), "direct path and pipeline kernel disagree"
    assert torch.equal(wire2, wire), "direct and pipeline payloads disagree"


def test_quantize_beyond_2_31_elements(oracle_mod):
    n, fmt = N_BIG, Q4
    x = long_message_bits(9300, n, F16)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    enc = torch.empty(qr.qr_encoded_bytes(fmt, n), dtype=torch.uint8, device="cuda")
    qr.qr_quantize(F16, fmt, xd, n, enc)
    torch.cuda.synchronize()
    blocks = boundary_blocks(n, 9301)
    sub = gather_blocks(x, blocks)
    o = oracle_mod.quantize(F16, fmt, sub)
    g_codes, g_scales, _ = split_encoded(enc.cpu().numpy(), fmt, n)
    o_codes, o_scales, _ = split_encoded(o, fmt, sub.size)
    assert np.array_equal(g_codes[blocks], o_codes)
    assert np.array_equal(g_scales[blocks], o_scales)
    # the direct encoder on the same message: the whole encoding bit for bit
    enc2 = torch.empty_like(enc)
    with qr.forced_kernel_path(qr.PATH_DIRECT):
        qr.qr_quantize(F16, fmt, xd, n, enc2)
        torch.cuda.synchronize()
    assert torch.equal(enc2, enc), "direct and pipeline encoders disagree"
