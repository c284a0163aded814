"""The bounds-checked library variant (libfp4moe_checked.so, compiled with
FP4MOE_BOUNDS_CHECK) on the GPU: the routing, permutation and MoE parity
tests run against it in a child process (the variant is chosen per process by
FP4MOE_BOUNDS_CHECK=1), where every call must leave the device status word at
OK, so no index check fires on valid inputs, and results still match the
oracle."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_the_bounds_checked_build():
    env = dict(os.environ, FP4MOE_BOUNDS_CHECK="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu",
           "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_kernels.py"),
           os.path.join(ROOT, "tests", "test_gpu_moe.py"),
           "-k", "route or permute or small_configs or token_counts or hot or "
                 "group32 or keep_group16 or index_check"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
