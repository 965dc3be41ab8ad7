"""The device path from a plain C program: tests/c/device_path.c, built with
the CUDA toolkit's compiler against include/moe.h and libmoe.so, allocates
its own device memory, runs moe_layout, moe_dispatch (FP8 records) and
moe_combine (grouped by rank) on inputs this test writes, then the one-call
layout + dispatch and the one-call fixed-capacity layout + dispatch
(moe_layout_ll_dispatch); its slot maps, records, combined rows, positions,
ranges and packed rows equal the oracle's."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from combine_moe_layout_03_gb300 import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "combine_moe_layout_03_gb300")


def test_c_program_runs_the_device_path(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cc = shutil.which("gcc") or shutil.which("cc")
    if not os.path.exists(nvcc) or cc is None:
        pytest.skip("no CUDA toolkit or C compiler")
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    cuda_lib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so")))
    from combine_moe_layout_03_gb300 import build
    build.build_library()
    exe = str(tmp_path / "device_path")
    subprocess.check_call([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "device_path.c"),
                           "-o", exe, "-L", PKG, "-lmoe", "-L", cuda_lib, "-lcudart",
                           f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{cuda_lib}"])

    c = synth.prefill_case(seed=31, n=512, hidden=1024)
    n, k, e, r, h = 512, 8, 256, 8, 1024
    ids, w, x = c["topk_idx"], c["topk_weights"], c["hidden_bf16"]
    lay = oracle.layout(ids, e, r)
    P = lay["num_pairs"]
    y = synth.bf16_normal(np.random.default_rng(32), (P, h))
    d = tmp_path / "io"
    d.mkdir()
    (d / "meta.txt").write_text(f"{n} {k} {e} {r} {h} {P}\n")
    ids.astype(np.int32).tofile(d / "ids.bin")
    w.astype(np.float32).tofile(d / "w.bin")
    x.astype(np.uint16).tofile(d / "x.bin")
    y.astype(np.uint16).tofile(d / "y.bin")
    run = subprocess.run([exe, str(d)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr

    slot = np.fromfile(d / "slot_of.bin", dtype=np.int32).reshape(n, k)
    np.testing.assert_array_equal(slot, lay["slot_of"])
    want = oracle.dispatch(ids, w, x, None, lay["slot_of"], P, oracle.BF16, oracle.FP8_E4M3_B128, h)
    got = np.fromfile(d / "records.bin", dtype=np.uint8).reshape(P, -1)
    np.testing.assert_array_equal(got, want)
    out = np.fromfile(d / "out.bin", dtype=np.uint16).reshape(n, h)
    np.testing.assert_array_equal(out, oracle.combine_topk_ranks(y, ids, w, lay["slot_of"], e, r, h))
    # the one-call form on the first 128 tokens (layout and dispatch in one kernel)
    ns = 128
    lay_s = oracle.layout(ids[:ns], e, r)
    ps = lay_s["num_pairs"]
    slot_s = np.fromfile(d / "slot_of_small.bin", dtype=np.int32).reshape(ns, k)
    np.testing.assert_array_equal(slot_s, lay_s["slot_of"])
    want_s = oracle.dispatch(ids[:ns], w[:ns], x[:ns], None, lay_s["slot_of"], ps, oracle.BF16,
                             oracle.FP8_E4M3_B128, h)
    got_s = np.fromfile(d / "records_small.bin", dtype=np.uint8).reshape(-1, got.shape[1])
    np.testing.assert_array_equal(got_s[:ps], want_s)

    # the fixed-capacity path on the first R * 16 tokens
    T = 16
    nl = r * T
    ll = oracle.ll_layout(ids[:nl], e, r, T)
    cap = r * T
    rows = e * cap
    np.testing.assert_array_equal(np.fromfile(d / "ll_slot_of.bin", dtype=np.int32).reshape(nl, k),
                                  ll["ll_slot_of"])
    np.testing.assert_array_equal(np.fromfile(d / "ll_src_info.bin", dtype=np.int32).reshape(e, cap),
                                  ll["src_info"])
    np.testing.assert_array_equal(np.fromfile(d / "ll_layout_range.bin", dtype=np.int64).reshape(e, r),
                                  ll["layout_range"])
    np.testing.assert_array_equal(np.fromfile(d / "ll_recv_count.bin", dtype=np.int32), ll["recv_count"])
    xo, so = oracle.dispatch_ll(x[:nl], None, ll["ll_slot_of"], rows, oracle.BF16, oracle.FP8_E4M3_B128, h)
    pos = ll["ll_slot_of"].ravel()
    used = pos >= 0
    assert used.all()                    # no pair past the capacity or without an expert here
    got_x = np.fromfile(d / "ll_x_pairs.bin", dtype=np.uint8).reshape(nl * k, xo.shape[1])
    got_s = np.fromfile(d / "ll_s_pairs.bin", dtype=np.uint8).reshape(nl * k, so.shape[1])
    np.testing.assert_array_equal(got_x, xo[pos])
    np.testing.assert_array_equal(got_s, so[pos])
