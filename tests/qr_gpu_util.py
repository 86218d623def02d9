"""Helpers shared by the GPU parity tests: device buffers with guard bands,
calls through the C ABI binding, and block sampling for full-size checks."""
import numpy as np
import torch

import quantized_allreduce_codec_gb300 as qr

GUARD = 256          # bytes of sentinel after every output buffer
SENTINEL = 0xA5


def dev_u16(bits: np.ndarray) -> torch.Tensor:
    """Host uint16 bit patterns -> device int16 tensor (16-byte aligned)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.cuda()


def host_u16(t: torch.Tensor, n: int) -> np.ndarray:
    return t[:n].cpu().numpy().view(np.uint16)


def out_buffer(nbytes: int) -> torch.Tensor:
    """A device byte buffer of nbytes plus a guard band, all set to SENTINEL."""
    return torch.full((nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")


def guard_intact(buf: torch.Tensor, nbytes: int) -> bool:
    return bool((buf[nbytes:] == SENTINEL).all().item())


def gpu_quantize(dtype, fmt, xb: np.ndarray):
    n = xb.size
    x = dev_u16(xb)
    nbytes = qr.qr_encoded_bytes(fmt, n)
    enc = out_buffer(nbytes)
    qr.qr_quantize(dtype, fmt, x, n, enc)
    torch.cuda.synchronize()
    assert guard_intact(enc, nbytes)
    return enc[:nbytes].cpu().numpy()


def gpu_dequantize(dtype, fmt, enc: np.ndarray, n: int):
    e = torch.from_numpy(np.ascontiguousarray(enc)).cuda()
    out = out_buffer(2 * n)
    qr.qr_dequantize(dtype, fmt, e, n, out)
    torch.cuda.synchronize()
    assert guard_intact(out, 2 * n)
    return out[:2 * n].cpu().numpy().view(np.uint16)


def gpu_allreduce(dtype, fmt, stages, xs, want_wire=True, dev_inputs=None):
    """Run qr_allreduce_emulated; returns (out bits, wire bytes or None)."""
    n = xs[0].size if xs is not None else dev_inputs[0].numel()
    ins = dev_inputs if dev_inputs is not None else [dev_u16(x) for x in xs]
    snap = [t.clone() for t in ins] if n <= (1 << 22) else None
    out = out_buffer(2 * n)
    wire = None
    wbytes = qr.qr_encoded_bytes(fmt, n)
    if stages == 2 and want_wire:
        wire = out_buffer(wbytes)
    qr.qr_allreduce_emulated(len(ins), dtype, fmt, stages, ins, n, out, wire)
    torch.cuda.synchronize()
    assert guard_intact(out, 2 * n)
    if wire is not None:
        assert guard_intact(wire, wbytes)
    if snap is not None:  # inputs are read only
        assert all(torch.equal(a, b) for a, b in zip(ins, snap))
    o = out[:2 * n].cpu().numpy().view(np.uint16)
    w = wire[:wbytes].cpu().numpy() if wire is not None else None
    return o, w


CODE_BITS = {1: 8, 2: 6, 3: 4, 4: 8, 5: 8, 6: 4}


def split_encoded(enc: np.ndarray, fmt: int, n: int):
    """(codes [nb, cb], scales [nb] uint16, zps [nb] uint16 or None)."""
    nb = (n + 31) // 32
    cb = 32 * CODE_BITS[fmt] // 8
    codes = enc[:nb * cb].reshape(nb, cb)
    scales = enc[nb * cb:nb * cb + 2 * nb].view(np.uint16)
    zps = enc[nb * cb + 2 * nb:nb * cb + 4 * nb].view(np.uint16) if fmt in (5, 6) else None
    return codes, scales, zps


def sample_blocks(n: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct block indices: first, last, tile edges and random ones."""
    nb = (n + 31) // 32
    rng = np.random.default_rng(seed)
    picks = {0, nb - 1, min(255, nb - 1), min(256, nb - 1), nb // 2}
    picks.update(rng.integers(0, nb, min(count, nb)).tolist())
    return np.array(sorted(picks), np.int64)


def gather_blocks(x: np.ndarray, blocks: np.ndarray) -> np.ndarray:
    """The elements of the given blocks, concatenated (a partial final block
    can only be the last one, so it stays last)."""
    n = x.size
    parts = [x[32 * b:min(32 * b + 32, n)] for b in blocks]
    return np.concatenate(parts)
