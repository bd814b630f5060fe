"""The bounds-checking debug build (compiled with KVQ_DEBUG_BOUNDS): every
index the kernels compute on the device is checked against its buffer, and
an index out of range would set KVQ_STATUS_BOUNDS (and skip the access)
rather than trap.  The option sweep of _bounds_sweep.py runs against that
build in a child process and must leave the status word at 0 and match the
oracle."""

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_option_sweep_under_the_debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_02_gb300 import build
    lib = build.build_debug()
    env = dict(os.environ, KVQ_LIB_PATH=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_bounds_sweep.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "bounds sweep ok" in r.stdout
