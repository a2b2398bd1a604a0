"""Host checks of numerical methods the kernels rely on (no GPU needed).

The q8_1 quantizer divides by 127 with one multiply and two fused
multiply-adds instead of an IEEE division; `host/div127_check.c` proves, with
the host's IEEE binary32 arithmetic, that the sequence returns the correctly
rounded quotient for every input the argument in its header does not cover by
scaling.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_division_by_127_is_correctly_rounded(tmp_path):
    exe = str(tmp_path / "div127_check")
    # no -ffast-math and no contraction: every operation is a single IEEE binary32 operation
    subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "host", "div127_check.c"), "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 mismatches" in r.stdout
