"""Index checks on the GPU: every entry point, on a library built with
-DKDA_CHECK_BOUNDS, leaves the status word clean (no global-memory index outside
its buffer).  Runs tests/bounds_run.py in a child process so that the checked
library is loaded on its own."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_no_index_leaves_its_buffer():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_run.py")], capture_output=True,
                         text=True, timeout=1200, cwd=ROOT)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "bounds ok" in out.stdout
