"""A bounded on-chip wait that runs out, without a fault.

Every mbarrier wait in the kernels is bounded (RS_DEV_PIPE_TIMEOUT).  The
program tests/c/wait_timeout.cu waits, through the library's own
mbar_wait_bounded, on a barrier that nothing arrives at: the wait must give
up after its poll limit, the kernel must report bit 8 in the status word and
return, and the context must stay usable for the next launch.  The measured
cycles per poll also give what the kernels' limit (kWaitPollLimit polls, then a
second bound) amounts to: about two seconds, not a hang.
"""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
DEVICE_HEADER = os.path.join(HERE, "..", "recurrent_state_gb300", "csrc", "rs_device.cuh")


def kernel_poll_limit():
    """kWaitPollLimit as the kernels are built with it."""
    with open(DEVICE_HEADER) as fh:
        m = re.search(r"kWaitPollLimit\s*=\s*1u\s*<<\s*(\d+)", fh.read())
    return 1 << int(m.group(1))


def test_wait_that_runs_out_reports_and_returns(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "wait_timeout")
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O2",
                           os.path.join(HERE, "c", "wait_timeout.cu"), "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = r.stdout.split("\n")
    runs = [tuple(int(x) for x in ln.split()) for ln in lines if ln and ln[0].isdigit()]
    assert len(runs) == 2
    for limit, status, cycles in runs:
        assert status == 8, (limit, status)
        assert cycles > 0
    assert "after ok" in r.stdout
    clock_khz = int([ln for ln in lines if ln.startswith("clock_khz")][0].split()[1]) or 2_070_000
    per_poll = runs[1][2] / runs[1][0]
    bound_s = 2 * kernel_poll_limit() * per_poll / (clock_khz * 1e3)
    print(f"cycles per poll {per_poll:.1f}; kernels' two bounds together ~{bound_s:.2f} s")
    # long enough for any copy of a stage (microseconds), short enough to report promptly
    assert 1e-2 < bound_s < 30
