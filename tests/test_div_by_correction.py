"""The attention backward forms a = p (/) l from RN(1/l) and two corrections by
fused multiply-add instead of a division per element (div2_rn in
csrc/k_attn.cuh).  This checks on the host's IEEE binary32 arithmetic (C99
fmaf rounds once) that the sequence returns the correctly rounded quotient,
bit for bit, over the ranges the kernel admits; outside them the kernel
divides.  The GPU side is covered by the attention parity tests."""
import pathlib
import shutil
import subprocess

import pytest


def test_quotient_by_correction_is_correctly_rounded(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = pathlib.Path(__file__).with_name("div_by_correction_check.c")
    exe = tmp_path / "div_check"
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-std=c11", "-o", str(exe), str(src), "-lm"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout
    assert "mismatches 0" in out.stdout, out.stdout
