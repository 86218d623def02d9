"""The direct kernel's block-scale reciprocal (two Newton-Raphson steps on the
hardware approximation) against the IEEE quotient 1/s that the method
defines, for every positive finite fp16 value s -- every block scale the
codec can produce.  numpy's float32 division is the IEEE round-to-nearest
quotient."""
import numpy as np
import pytest
import torch

import quantized_allreduce_codec_gb300 as qr
from quantized_allreduce_codec_gb300 import build

pytestmark = pytest.mark.gpu


def test_reciprocal_of_every_fp16_scale_is_the_ieee_quotient():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    out = torch.full((qr.SELFTEST_RECIPROCALS,), float("nan"), dtype=torch.float32, device="cuda")
    qr.qr_selftest_reciprocal(out)
    torch.cuda.synchronize()
    s = np.arange(1, qr.SELFTEST_RECIPROCALS + 1, dtype=np.uint16).view(np.float16).astype(np.float32)
    assert np.isfinite(s).all() and s.max() == np.float32(65504.0) and s.min() == np.float32(2.0 ** -24)
    want = (np.float32(1.0) / s).view(np.uint32)
    got = out.cpu().numpy().view(np.uint32)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(s[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]
