"""The mixed decode kernel forms the INT8 row scale RN(max(a, 1e-8) / 127)
without a division (q0 = RN(a * RN(1/127)) plus one exact-remainder
correction, Markstein's step).  This checks the identity for every finite FP32
input the kernel can see (a >= 1e-8), on the CPU, with each operation rounded
once (DAMP §3.2 Eq. 5, dasc Appendix E.1 Eq. 8: s = max(absmax, 1e-8) / 127)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_division_free_scale_is_exact_for_every_input(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "div127")
    subprocess.check_call([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           os.path.join(HERE, "c", "div127_exhaustive.c"), "-o", exe, "-lm"])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    n, bad = map(int, r.stdout.split())
    assert n == 1297363849  # every finite float from 1e-8 up
    assert bad == 0 and r.returncode == 0
