"""The checked build (-DDSA_CHECKS=1) reports out-of-range device-side inputs (GPU).

The library to load is chosen at its first load, so the case runs in a process of its
own (tests/checked_build_case.py) with DSA_CHECKED=1."""
import os
import subprocess
import sys

import pytest
import torch

from dynamic_sparse_attention_gb300 import _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_bad_device_inputs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    _build.build(checked=True)
    env = dict(os.environ, DSA_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_build_case.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked-build ok" in r.stdout
