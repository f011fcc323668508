"""The opt-in single-read quantize against the same bar as the default path.

By default a quantize call runs two launches: the column-statistics pass,
then the quantize pass.  With ``AVERIS_SINGLE_READ_QUANTIZE=1`` (read when
the library first sees the device), tensors whose 128 x 128 tiles all fit the
resident CTAs' buffers, without the Hadamard rotation, take one cooperative
launch that reads X once and keeps its tiles in shared memory.  This runs the
quantize parity, timeout and linear-layer tests again in a child process with
it set: both paths meet the same bar on the same small and ragged shapes.
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_quantize_parity_on_the_single_read_path(cuda_lib):
    env = dict(os.environ, AVERIS_SINGLE_READ_QUANTIZE="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_quant.py", "tests/test_gpu_timeout.py", "tests/test_gpu_linear.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_single_read_path_under_the_bounds_checks(cuda_lib):
    """The debug build's tiny-shape run (every computed address checked, see
    test_gpu_debug_bounds.py) with the single-read launch taking every quantize
    call that it can, so that its partials and mean stores are checked too."""
    env = dict(os.environ, AVERIS_SINGLE_READ_QUANTIZE="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_debug_bounds.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
