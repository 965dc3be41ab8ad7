"""The top-k combine has three kernels: a persistent warp-per-slice kernel, a
block-per-row kernel, and a pipelined kernel whose expert rows reach shared
memory through bulk copies. moe_combine picks one by size; the environment
variable MOE_COMBINE_PIPE (read once per process) overrides that: 0 never
takes the pipelined kernel, 2 takes it at every size. The combine parity
files pass in child processes under both settings, so each kernel meets the
oracle on every shape those files draw. Runs of the pipelined kernel leave
the library's device status word at MOE_OK (no bounded wait gave up). With
the waits' budget lowered to 1 ns (moe_set_wait_limit_ns) the pipelined
kernel's waits give up: the status word reads MOE_ERR_TIMEOUT, and the same
call with the default budget afterwards, in the same context, is bit-exact
against the oracle."""
import os
import subprocess
import sys

import pytest
import torch

import numpy as np

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, host_bf16

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


@pytest.mark.skipif(os.environ.get("MOE_COMBINE_PIPE") == "0", reason="the pipelined kernel is switched off")
def test_bounded_waits_give_up_and_the_context_stays_usable():
    from combine_moe_layout_03_gb300 import moe
    # 4 ranks x 64 tokens, H=8192, top-8 of 256 grouped by rank: a shape the
    # automatic choice sends to the pipelined kernel
    n, k, e, r, h = 256, 8, 256, 4, 8192
    c = synth.rs_case(seed=17, tokens_per_rank=64, hidden=h, r=r, e=e, k=k, with_partials=False)
    ids, w, y = c["topk_idx"], c["topk_weights"], c["expert_out_bf16"]
    d = moe.MoeDesc(n, k, e, r, h)
    ids_d, w_d, y_d = dev_i32(ids), dev_f32(w), dev_bf16(y)
    lay = moe.moe_layout(d, ids_d)
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=True) == moe.MOE_OK
    try:
        moe.moe_set_wait_limit_ns(1)
        moe.moe_combine(d, moe.MOE_COMBINE_TOPK_RANKS, y_d, ids_d, w_d, lay["slot_of"])
        assert moe.moe_device_status(clear=True) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_set_wait_limit_ns(0)
    out = moe.moe_combine(d, moe.MOE_COMBINE_TOPK_RANKS, y_d, ids_d, w_d, lay["slot_of"])
    torch.cuda.synchronize()
    assert moe.moe_device_status(clear=True) == moe.MOE_OK
    ref = oracle.layout(ids, e, r)
    want = oracle.combine_topk_ranks(y, ids, w, ref["slot_of"], e, r, h)
    np.testing.assert_array_equal(host_bf16(out), want)
