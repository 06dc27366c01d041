"""The checks build on the GPU.

libvw4_checks.so is the library compiled with -DVW4_CHECKS: its kernels test
the indexes that come from data (the output row a MoE routing table names,
the activation row a segment reads, the token ids an accept commits) and
report a failed test as VW4_DEV_BOUNDS in the device status word.  The guard
canary suite (every entry point, every output), the MoE suite and the fused
accept suite run in a child process against it; they check parity and a zero
device status after every call, so they pass only if no check failed.
"""
import os
import subprocess
import sys

import pytest

from speculative_decode_verification_w4_gb300 import build as vbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_canaries_gpu.py", "tests/test_moe_gpu.py", "tests/test_fused_accept_gpu.py"]


def test_checks_build_passes_the_canary_moe_and_fused_accept_suites():
    path = vbuild.build(checks=True)
    env = dict(os.environ, VW4_LIB=path)
    probe = subprocess.run(
        [sys.executable, "-c", "import speculative_decode_verification_w4_gb300 as v; "
                               "print(v.vw4_build_flags())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip() == "1", probe.stdout   # the child loads the checks build
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                        "-p", "no:cacheprovider", *SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
