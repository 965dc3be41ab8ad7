"""The C ABI from plain C: a C11 program (tests/c/host_abi.c) compiles
against include/moe.h with warnings as errors, links libmoe.so, and its
host-only calls give the oracle's record layout, a usable workspace size,
named argument errors and a record that packs and unpacks unchanged. No GPU
is needed: these entry points never touch the device."""
import os
import shutil
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "combine_moe_layout_03_gb300")


def _run(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from combine_moe_layout_03_gb300 import build
    build.build_library()
    exe = str(tmp_path / "host_abi")
    subprocess.check_call([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "host_abi.c"), "-o", exe, "-L", PKG, "-lmoe",
                           f"-Wl,-rpath,{PKG}"])
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    return dict(line.split("=", 1) for line in out.splitlines())


def test_c_program_uses_the_host_entry_points(tmp_path):
    kv = _run(tmp_path)
    assert kv["fp8_rc"] == "0"
    want = oracle.record_layout(8, 7168, oracle.BF16, oracle.FP8_E4M3_B128)
    for key in ("record_bytes", "off_ids", "off_weights", "off_payload", "off_scales", "payload_bytes",
                "scale_bytes"):
        assert int(kv["fp8_" + key]) == int(want[key]), key
    assert int(kv["fp8_record_bytes"]) == 7472  # the prefill record size of the pages' formula
    assert int(kv["workspace_bytes"]) >= 256
    assert int(kv["bad_ranks_rc"]) < 0 and kv["bad_ranks_name"]
    assert int(kv["null_desc_rc"]) < 0
    assert kv["bf16_rc"] == "0" and kv["pack_rc"] == "0" and kv["unpack_rc"] == "0"
    assert (kv["src_token"], kv["slot_j"], kv["expert"]) == ("3", "1", "11")
    assert kv["ids_equal"] == kv["weights_equal"] == kv["row_equal"] == "1"
