"""The bounds-checked debug build on the GPU: the library compiled with -DFTMOE_CHECK tests
device-side indices (miss list, copy targets, FFN slots) before using them and records a status
code instead of touching memory out of bounds. Parity tests covering every pipeline run in a
child process that loads that build (FTMOE_CHECKED=1) and must pass unchanged: no check fires
on correct inputs, and results are the same."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_under_the_bounds_checked_build():
    from expert_slot_cache_device_gb300 import build

    build.build(check=True)
    env = dict(os.environ, FTMOE_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_parity.py"),
           "-k", "small_geometries or combine_edge or kernel_families or random_traces or error_paths"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
