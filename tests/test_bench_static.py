"""Static checks of the host scripts that only a GPU run executes end to end:
every global name a function of bench.py, __graft_entry__.py or the Python
binding reads is defined at module level or is a builtin (a misplaced
variable in a rarely run branch otherwise shows up first on the GPU)."""
import builtins
import os
import symtable

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["bench.py", "__graft_entry__.py", os.path.join("combine_moe_layout_03_gb300", "moe.py")]


def _undefined_globals(path):
    src = open(path).read()
    top = symtable.symtable(src, path, "exec")
    defined = set(top.get_identifiers())
    bad = []

    def walk(t):
        for ch in t.get_children():
            if ch.get_type() == "function":
                for sym in ch.get_symbols():
                    name = sym.get_name()
                    if (sym.is_global() and sym.is_referenced() and name not in defined
                            and not hasattr(builtins, name)):
                        bad.append(f"{ch.get_name()}: {name}")
            walk(ch)

    walk(top)
    return bad


@pytest.mark.parametrize("rel", FILES)
def test_no_undefined_global_names(rel):
    assert _undefined_globals(os.path.join(ROOT, rel)) == []
