"""The kernels' bounded waits, made to run out on purpose: a barrier that
nothing completes, a short limit, and the flag the host reads afterwards.
No fault, no trap, no hang: the kernel returns on its own."""
import time

import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qr.lib()
    qr.qr_device_error(clear=True)


def test_wait_gives_up_and_raises_flag():
    t0 = time.perf_counter()
    qr.qr_selftest_wait_timeout(20000)  # 20 ms
    flags = qr.qr_device_error(clear=True)
    elapsed = time.perf_counter() - t0
    assert flags == 8
    assert 0.015 < elapsed < 5.0
    assert qr.qr_device_error(clear=True) == 0  # cleared


def test_context_still_usable_after_timeout():
    qr.qr_selftest_wait_timeout(1000)
    assert qr.qr_device_error(clear=True) == 8
    x = torch.ones(4096, dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    qr.qr_allreduce_emulated(2, qr.F16, qr.QR_FP, 1, [x, x], x.numel(), out)
    torch.cuda.synchronize()
    assert torch.all(out == 2).item()
    assert qr.qr_device_error(clear=True) == 0


def test_limit_out_of_range():
    with pytest.raises(qr.QRError, match="QR_ERR_SIZE"):
        qr.qr_selftest_wait_timeout(0)
    with pytest.raises(qr.QRError, match="QR_ERR_SIZE"):
        qr.qr_selftest_wait_timeout(2000000)
