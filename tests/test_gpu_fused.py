"""moe_layout_dispatch (layout and dispatch in one call, the dispatch's row
work overlapping the layout) gives the oracle's layout and records bit for
bit, for every payload format and the edge cases; a bad dispatch argument is
rejected before the layout is launched."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_layout_03_gb300 import synth

from gpu_helpers import DEV, dev_bf16, dev_f32, dev_i32, dev_u8, host

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("tokens_per_expert", "tokens_per_rank", "is_token_in_rank", "expert_offset",
               "rank_offset", "slot_of")


def _check(c, e, r, in_kind, out_kind, x_host, x_dev, sc_host=None, sc_dev=None, rp=0, rs=0,
           sample=None):
    from combine_moe_layout_03_gb300 import moe
    ids, w = c["topk_idx"], c["topk_weights"]
    n, k = ids.shape
    d = moe.MoeDesc(n, k, e, r, c["hidden"], in_kind, out_kind, rp, rs)
    rb = moe.moe_record_layout(d)["record_bytes"]
    rec = torch.full((n * k + 2, rb), 0xAB, dtype=torch.uint8, device=DEV)
    lay, rec = moe.moe_layout_dispatch(d, dev_i32(ids), dev_f32(w), x_dev, sc_dev, records=rec)
    torch.cuda.synchronize()
    ref = oracle.layout(ids, e, r)
    for key in LAYOUT_KEYS:
        np.testing.assert_array_equal(host(lay[key]).reshape(ref[key].shape), ref[key], err_msg=key)
    P = ref["num_pairs"]
    got = host(rec)
    assert np.all(got[P:] == 0xAB)
    if sample is None:
        want = oracle.dispatch(ids, w, x_host, sc_host, ref["slot_of"], P, in_kind, out_kind,
                               c["hidden"], rp, rs)
        np.testing.assert_array_equal(got[:P], want)
        return
    for t0, t1 in sample:
        sub = slice(t0, t1)
        want = oracle.dispatch(ids[sub], w[sub], x_host[sub], None if sc_host is None else sc_host[sub],
                               ref["slot_of"][sub], P, in_kind, out_kind, c["hidden"], rp, rs)
        slots = ref["slot_of"][sub].ravel()
        slots = slots[slots >= 0]
        rows = want[slots].copy()
        rows[:, :4].view(np.int32)[:] += t0  # the oracle numbered the sub-range from 0
        np.testing.assert_array_equal(got[slots], rows)


def test_fused_prefill_fp8_full_size_sampled():
    c = synth.prefill_case(seed=90)
    _check(c, 256, 8, oracle.BF16, oracle.FP8_E4M3_B128, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]),
           sample=[(0, 32), (2000, 2048), (4064, 4096)])


def test_fused_decode_raw():
    c = synth.decode_case(seed=91, n=256)
    _check(c, 256, 8, oracle.RAW, oracle.RAW, c["payload"], dev_u8(c["payload"]), c["scales"],
           dev_u8(c["scales"]), 3584, 448)


@pytest.mark.parametrize("out_kind", [oracle.BF16, oracle.NVFP4_B16])
def test_fused_small_formats(out_kind):
    c = synth.prefill_case(seed=92, n=100, hidden=1024)
    c["topk_idx"] = c["topk_idx"].copy()
    c["topk_idx"][::7, 3] = -1
    _check(c, 256, 8, oracle.BF16, out_kind, c["hidden_bf16"], dev_bf16(c["hidden_bf16"]))


def test_fused_two_kernel_layout_shape():
    # a shape whose layout takes the two-kernel path (cluster shared memory too big)
    g = np.random.default_rng(93)
    n, k, e, r, h = 90000, 8, 512, 16, 128
    ids = np.stack([g.permutation(e)[:k] for _ in range(n)]).astype(np.int32)
    c = dict(topk_idx=ids, topk_weights=g.standard_normal((n, k)).astype(np.float32), hidden=h)
    x = synth.bf16_normal(g, (n, h))
    _check(c, e, r, oracle.BF16, oracle.FP8_E4M3_B128, x, dev_bf16(x),
           sample=[(0, 16), (45000, 45016), (89984, 90000)])


def test_fused_empty_batch():
    from combine_moe_layout_03_gb300 import moe
    d = moe.MoeDesc(0, 8, 256, 8, 7168, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    ids = torch.empty((0, 8), dtype=torch.int32, device=DEV)
    w = torch.empty((0, 8), dtype=torch.float32, device=DEV)
    x = torch.empty((0, 7168), dtype=torch.bfloat16, device=DEV)
    rec = torch.full((4, 7472), 0xAB, dtype=torch.uint8, device=DEV)
    lay, rec = moe.moe_layout_dispatch(d, ids, w, x, None, records=rec)
    torch.cuda.synchronize()
    assert (host(lay["tokens_per_expert"]) == 0).all() and (host(lay["expert_offset"]) == 0).all()
    assert (host(rec) == 0xAB).all()


def test_fused_rejects_bad_dispatch_argument_before_the_layout():
    from combine_moe_layout_03_gb300 import moe
    c = synth.prefill_case(seed=94, n=64, hidden=1024)
    d = moe.MoeDesc(64, 8, 256, 8, 1024, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    lay = {key: torch.full_like(v, 77) for key, v in moe.layout_outputs(d, DEV).items()}
    ws = torch.empty(max(moe.moe_workspace_size(d), 256), dtype=torch.uint8, device=DEV)
    small = torch.empty((1, 64), dtype=torch.uint8, device=DEV)  # smaller than one record
    with pytest.raises(RuntimeError):
        moe.prepare_layout_dispatch(d, dev_i32(c["topk_idx"]), dev_f32(c["topk_weights"]),
                                    dev_bf16(c["hidden_bf16"]), None, lay, ws, small)()
    torch.cuda.synchronize()
    assert (host(lay["slot_of"]) == 77).all()  # the layout did not run


@pytest.mark.parametrize("out_kind,hidden,n", [
    (oracle.FP8_E4M3_B128, 128, 37),      # one group: a partial wave of one half-warp
    (oracle.FP8_E4M3_B128, 1152, 300),    # nine groups: a full wave and a partial one
    (oracle.FP8_E4M3_B128, 7168, 64),
    (oracle.FP8_E4M3_B128, 16384, 40),    # largest hidden size
    (oracle.NVFP4_B16, 16, 50),           # one group of 16
    (oracle.NVFP4_B16, 48, 50),
    (oracle.NVFP4_B16, 1040, 120),
    (oracle.NVFP4_B16, 7168, 64),
    (oracle.NVFP4_B16, 16384, 40),
    (oracle.FP8_E4M3_UE8M0, 128, 37),
    (oracle.FP8_E4M3_UE8M0, 7168, 64),
    (oracle.FP8_E4M3_UE8M0, 16384, 40),
])
def test_fused_quantised_rows_every_width(out_kind, hidden, n):
    """The fused call quantises each row in place in its record image; every
    record of every width must still equal the oracle's."""
    c = synth.prefill_case(seed=hidden + n, n=n, hidden=hidden)
    x = c["hidden_bf16"].copy()
    x[0] = 0                        # an all-zero row
    x[1, : min(hidden, 128)] = 0x7F7F  # the largest finite BF16
    x[2, ::3] = 0x8000               # negative zeros
    x[3, : min(hidden, 64)] = 0x0001  # subnormals
    c["hidden_bf16"] = x
    _check(c, 256, 8, oracle.BF16, out_kind, x, dev_bf16(x))
