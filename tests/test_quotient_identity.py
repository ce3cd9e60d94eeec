"""The page-quantise kernel's quotient without a division, checked on the host.

The handoff quantiser replaces the append rule's IEEE fp32 division x / s by
a multiplication with RN(1 / s) and one fused multiply-add correction
(Markstein's step), after clamping x to +-1024 s.  quotient_identity.c checks,
in C float arithmetic with fmaf, that this gives RN(x / s) for every bf16
significand against every fp32 significand of the scale, and that the clamp
and the scale range [2^-90, 2^100] keep every e4m3 decision the same for all
bf16 bit patterns.  The GPU tests compare the kernel's codes with the oracle
over all bf16 values as well."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_corrected_quotient_equals_ieee_division(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "quotient_identity"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-o", str(exe),
                    os.path.join(HERE, "quotient_identity.c"), "-lm"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout
    assert "mismatches 0" in out.stdout
