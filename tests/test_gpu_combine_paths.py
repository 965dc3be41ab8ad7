"""The top-k combine has three kernels: a persistent warp-per-slice kernel, a
block-per-row kernel, and a pipelined kernel whose expert rows reach shared
memory through bulk copies. moe_combine picks one by size; the environment
variable MOE_COMBINE_PIPE (read once per process) overrides that: 0 never
takes the pipelined kernel, 2 takes it at every size. The combine parity
files pass in child processes under both settings, so each kernel meets the
oracle on every shape those files draw. Runs of the pipelined kernel leave
the library's device status word at MOE_OK (no bounded wait gave up)."""
import os
import subprocess
import sys

import pytest
import torch

from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
FILES = ["test_gpu_combine.py", "test_gpu_random_shapes.py", "test_gpu_ll.py", "test_gpu_backward.py"]


@pytest.mark.parametrize("policy", ["0", "2"])
def test_combine_parity_files_under_each_kernel_choice(policy):
    env = dict(os.environ, MOE_COMBINE_PIPE=policy)
    run = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                          *[os.path.join(HERE, f) for f in FILES]],
                         env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True, timeout=1200)
    assert run.returncode == 0, run.stdout[-3000:] + run.stderr[-2000:]
    assert " passed" in run.stdout


def test_device_status_stays_ok_after_pipelined_combines():
    from combine_moe_layout_03_gb300 import moe
    assert moe.moe_device_status(clear=True) == moe.MOE_OK
    for n, mode in ((1, moe.MOE_COMBINE_TOPK), (64, moe.MOE_COMBINE_TOPK_RANKS), (256, moe.MOE_COMBINE_TOPK_RANKS)):
        c = synth.decode_case(seed=n, n=n)
        d = moe.MoeDesc(n, 8, 256, 8, 7168)
        ids = dev_i32(c["topk_idx"])
        lay = moe.moe_layout(d, ids)
        y = dev_bf16(synth.bf16_normal(synth.rng_for(n, 3), (n * 8, 7168)))
        moe.moe_combine(d, mode, y, ids, dev_f32(c["topk_weights"]), lay["slot_of"])
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=False) == moe.MOE_OK
