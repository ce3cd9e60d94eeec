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


def _run(tmp_path, *defines):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "quotient_identity"
    subprocess.run([cc, "-O2", "-ffp-contract=off", *defines, "-o", str(exe),
                    os.path.join(HERE, "quotient_identity.c"), "-lm"], check=True)
    return subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)


def test_corrected_quotient_equals_ieee_division(tmp_path):
    out = _run(tmp_path)
    assert out.returncode == 0, out.stdout
    assert "mismatches 0" in out.stdout


def test_check_fails_without_the_correction(tmp_path):
    """The same check on the uncorrected product x * RN(1 / s) must find
    mismatches (over 900,000 of the 40 M cases of this reduced run): it is
    not vacuous."""
    out = _run(tmp_path, "-DQI_DROP_CORRECTION", "-DQI_SCALE_SIGNIFICANDS=4096u")
    assert out.returncode == 1
    bad = int(out.stdout.split("mismatches")[-1])
    assert bad > 10000
