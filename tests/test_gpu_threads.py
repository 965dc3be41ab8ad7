"""Calls from several host threads at once, each on its own stream, give the
same results as one thread: the library keeps no per-call host state and its
per-device caches are filled once under a lock."""
import threading

import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, host, host_bf16

pytestmark = pytest.mark.gpu


def test_concurrent_host_threads_on_separate_streams():
    from combine_moe_layout_03_gb300 import moe
    cases = [synth.prefill_case(seed=80 + i, n=256 + 64 * i, hidden=1024) for i in range(4)]
    results, errors = [None] * 4, []

    def work(i):
        try:
            c = cases[i]
            n = c["topk_idx"].shape[0]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                d = moe.MoeDesc(n, 8, 256, 8, 1024, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
                ids = dev_i32(c["topk_idx"])
                lay = moe.moe_layout(d, ids, stream=s.cuda_stream)
                rec = moe.moe_dispatch(d, ids, dev_f32(c["topk_weights"]), dev_bf16(c["hidden_bf16"]),
                                       None, lay["slot_of"], stream=s.cuda_stream)
            s.synchronize()
            results[i] = (host(lay["slot_of"]), host(rec))
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i, c in enumerate(cases):
        lay = oracle.layout(c["topk_idx"], 256, 8)
        np.testing.assert_array_equal(results[i][0], lay["slot_of"])
        P = lay["num_pairs"]
        ref = oracle.dispatch(c["topk_idx"], c["topk_weights"], c["hidden_bf16"], None, lay["slot_of"], P,
                              oracle.BF16, oracle.FP8_E4M3_B128, 1024)
        np.testing.assert_array_equal(results[i][1][:P], ref)
