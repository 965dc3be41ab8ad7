"""With MOE_FUSED_LAYOUT=0 moe_layout_dispatch keeps the layout kernel and
the early dispatch at every size: the small-routing parity file
(tests/test_gpu_fused_small.py) passes on that path too, in a child process
(the switch is read once per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_small_routings_on_the_two_kernel_path():
    env = dict(os.environ, MOE_FUSED_LAYOUT="0")
    run = subprocess.run([sys.executable, "-m", "pytest", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                          os.path.join(HERE, "test_gpu_fused_small.py")],
                         env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=600)
    assert run.returncode == 0, run.stdout[-3000:] + run.stderr[-2000:]
    assert " passed" in run.stdout
