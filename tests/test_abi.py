"""The C-ABI library loads, exports every entry point include/moe.h declares,
and its host-only logic (record layout, pack/unpack, argument validation)
behaves as documented. No compute calls: these run without a GPU."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from combine_moe_layout_03_gb300 import build
    build.build_library()
    from combine_moe_layout_03_gb300 import moe as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("moe_layout", "moe_dispatch", "moe_combine", "moe_pack_record",
                 "moe_unpack_record", "moe_record_layout", "moe_workspace_size", "moe_strerror",
                 "moe_layout_status"):
        assert must in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(_declared_functions()) <= exported
    assert set(moe.exported_symbols()) == set(_declared_functions())


def _golden_rows():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "record_sizes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            name, *vals = line.split()
            rows.append((name, *map(int, vals)))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_record_layout_matches_page_formulas(moe, row):
    name, k, h, ik, ok, rp, rs, rec_bytes, body = row
    lay = moe.moe_record_layout(moe.MoeDesc(16, k, 256, 8, h, ik, ok, rp, rs))
    assert lay["record_bytes"] == rec_bytes
    pad = lambda x: (x + 15) // 16 * 16
    assert rec_bytes - 16 - 2 * pad(4 * k) == body
    assert all(lay[key] % 16 == 0 for key in ("off_ids", "off_weights", "off_payload",
                                              "off_scales", "record_bytes"))


def test_pack_unpack_round_trip(moe):
    d = moe.MoeDesc(4, 3, 12, 3, 128, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128)
    g = np.random.default_rng(0)
    ids = np.array([7, -1, 2], np.int32)
    w = np.array([0.5, 0.25, -1.5], np.float32)
    pay = g.integers(0, 256, 128, dtype=np.uint8)
    sc = np.frombuffer(np.float32([1.5 / 448]).tobytes(), np.uint8)
    rec = moe.moe_pack_record(d, 3, 2, 2, ids, w, pay, sc)
    lay = moe.moe_record_layout(d)
    assert rec.size == lay["record_bytes"]
    u = moe.moe_unpack_record(d, rec)
    assert (u["src_token"], u["slot_j"], u["expert"]) == (3, 2, 2)
    np.testing.assert_array_equal(u["ids"], ids)
    np.testing.assert_array_equal(u["weights"], w)
    np.testing.assert_array_equal(u["payload"], pay)
    np.testing.assert_array_equal(u["scales"], sc)
    assert rec[12:16].tolist() == [0, 0, 0, 0]
    used = np.zeros(rec.size, bool)
    used[:12] = True
    for off, n in ((lay["off_ids"], 12), (lay["off_weights"], 12),
                   (lay["off_payload"], lay["payload_bytes"]), (lay["off_scales"], lay["scale_bytes"])):
        used[off:off + n] = True
    assert np.all(rec[~used] == 0)


def test_pack_record_layout_agrees_with_byte_offsets(moe):
    # The header's int32 fields sit at bytes 0, 4, 8 (little-endian).
    d = moe.MoeDesc(2, 2, 4, 2, 16)
    rec = moe.moe_pack_record(d, 0x01020304, 1, 3, np.int32([3, 1]), np.float32([1, 2]),
                              np.arange(32, dtype=np.uint8), None)
    assert rec[:4].tolist() == [4, 3, 2, 1]
    assert rec[4:8].view(np.int32)[0] == 1 and rec[8:12].view(np.int32)[0] == 3


@pytest.mark.parametrize("kwargs,code", [
    (dict(num_experts=10, num_ranks=4), -3),   # E % R
    (dict(topk=33), -3),                       # k > 32
    (dict(num_ranks=65, num_experts=130), -3), # R > 64
    (dict(num_experts=2048), -3),              # E > 1024
    (dict(num_tokens=-1), -3),
    (dict(topk=0), -3),
])
def test_shape_errors_return_codes_without_launch(moe, kwargs, code):
    base = dict(num_tokens=8, topk=2, num_experts=8, num_ranks=2, hidden=64)
    base.update(kwargs)
    d = moe.MoeDesc(**base)
    assert moe.moe_workspace_size(d) == 0
    rc = moe._lib.moe_layout(ctypes.byref(d.c()), 16, 16, 16, 16, 16, 16, 16, None, 256, 1 << 20,
                             None)
    assert rc == code


def test_argument_errors_return_codes_without_launch(moe):
    d = moe.MoeDesc(8, 2, 8, 2, 64)
    c = d.c()
    ws = moe.moe_workspace_size(d)
    assert ws > 0 and ws % 256 == 0
    lib = moe._lib
    # NULL output
    assert lib.moe_layout(ctypes.byref(c), 16, None, 16, 16, 16, 16, 16, None, 256, ws, None) == -1
    # misaligned int pointer, misaligned workspace, workspace too small
    assert lib.moe_layout(ctypes.byref(c), 18, 16, 16, 16, 16, 16, 16, None, 256, ws, None) == -2
    assert lib.moe_layout(ctypes.byref(c), 16, 16, 16, 16, 16, 16, 16, None, 272, ws, None) == -2
    assert lib.moe_layout(ctypes.byref(c), 16, 16, 16, 16, 16, 16, 16, None, 256, ws - 1, None) == -4
    # dispatch: bad kind pair, misaligned records, too small a records buffer
    bad = moe.MoeDesc(8, 2, 8, 2, 64, moe.MOE_PAYLOAD_RAW, moe.MOE_PAYLOAD_BF16).c()
    assert lib.moe_dispatch(ctypes.byref(bad), 16, 16, 16, None, 16, 16, 1 << 20, None) == -1
    assert lib.moe_dispatch(ctypes.byref(c), 16, 16, 16, None, 16, 24, 1 << 20, None) == -2
    assert lib.moe_dispatch(ctypes.byref(c), 16, 16, 16, None, 16, 32, 64, None) == -4
    # FP8 needs H % 128; RAW needs 16-byte multiples
    f8 = moe.MoeDesc(8, 2, 8, 2, 64, moe.MOE_PAYLOAD_BF16, moe.MOE_PAYLOAD_FP8_E4M3_B128).c()
    assert lib.moe_dispatch(ctypes.byref(f8), 16, 16, 16, None, 16, 32, 1 << 20, None) == -3
    raw = moe.MoeDesc(8, 2, 8, 2, 64, moe.MOE_PAYLOAD_RAW, moe.MOE_PAYLOAD_RAW, 100, 0).c()
    assert lib.moe_dispatch(ctypes.byref(raw), 16, 16, 16, None, 16, 32, 1 << 20, None) == -2
    # combine: bad mode, H % 8, N % R for the rank modes, capacity of partials
    assert lib.moe_combine(ctypes.byref(c), 7, 16, 100, 16, 16, 16, 16, None) == -1
    h7 = moe.MoeDesc(8, 2, 8, 2, 7).c()
    assert lib.moe_combine(ctypes.byref(h7), 0, 16, 100, 16, 16, 16, 16, None) == -3
    odd = moe.MoeDesc(7, 2, 8, 2, 64).c()
    assert lib.moe_combine(ctypes.byref(odd), 1, 16, 100, None, None, None, 16, None) == -3
    assert lib.moe_combine(ctypes.byref(c), 1, 16, 15, None, None, None, 16, None) == -4
    assert lib.moe_combine(ctypes.byref(c), 2, 16, 100, None, 16, 16, 16, None) == -1


def test_strerror_covers_codes(moe):
    for code in range(0, -9, -1):
        assert moe.moe_strerror(code) != "unknown status"
    assert moe.moe_strerror(-99) == "unknown status"
