"""The kernels divide by the format's level count with a reciprocal and one
exact-remainder correction instead of an IEEE divide.  This checks, on the
CPU in C, that the fp16 scale it yields equals the one from IEEE division
for non-negative binary32 inputs: every exponent with a stride through the
mantissas by default, every value with QR_EXHAUSTIVE=1 (about 3 minutes)."""
import os
import platform
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_scale_division_matches_ieee(tmp_path):
    exe = tmp_path / "scale_division_check"
    flags = ["-O2", "-ffp-contract=off", "-fno-fast-math"]
    if platform.machine() in ("x86_64", "AMD64"):
        flags.append("-mfma")  # hardware FMA; fmaf is exact either way
    subprocess.run(["gcc", *flags, "-o", str(exe), os.path.join(HERE, "scale_division_check.c"), "-lm"],
                   check=True)
    stride = "0" if os.environ.get("QR_EXHAUSTIVE") == "1" else "9"
    r = subprocess.run([str(exe), stride], capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.strip().splitlines()
    assert len(lines) == 6
    for ln in lines:
        fields = dict(kv.split("=") for kv in ln.split())
        assert int(fields["scale_mismatch"]) == 0, ln
        if fields["L"] != "448":  # 448: mismatches only far below the fp16 range
            assert int(fields["quotient_mismatch"]) == 0, ln
        else:
            assert float(fields["max_mismatch_quotient"]) < 2.0 ** -100, ln
