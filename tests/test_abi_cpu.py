"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point declared in include/gattn.h, and rejects bad arguments on
the host before touching CUDA.  No compute call is made."""
import ctypes
import os
import re

import pytest

from gnn_sparse_attention_gb300 import binding as gb
from gnn_sparse_attention_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gb.load_library()


def _declared():
    with open(os.path.join(ROOT, "include", "gattn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"GATTN_API\s+[\w\s\*]*?\b(gattn_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = _declared()
    assert set(names) == set(gb.EXPORTED), names


def test_library_exports_every_declared_symbol(lib):
    out = os.popen(f"nm -D --defined-only {gb.library_path()}").read()
    exported = set(re.findall(r"\sT\s+(gattn_\w+)", out))
    missing = set(_declared()) - exported
    assert not missing, missing
    for name in _declared():
        assert hasattr(lib, name)


def test_version(lib):
    assert gb.gattn_version().startswith("gattn ")
    assert "sm_103a" in gb.gattn_version()


def test_host_argument_checks(lib):
    h = ctypes.c_void_p()
    assert lib.gattn_plan_create(None, None, 4, 0, None, None, None) == 1
    assert b"out is NULL" in lib.gattn_last_error()
    assert lib.gattn_plan_create(None, None, -1, 0, None, None, ctypes.byref(h)) == 1
    assert lib.gattn_plan_create(None, None, 4, 1 << 31, None, None, ctypes.byref(h)) == 1
    assert lib.gattn_plan_create(None, None, 4, 0, None, None, ctypes.byref(h)) == 1
    assert h.value is None
    assert lib.gattn_plan_get_info(None, None) == 1
    assert lib.gattn_plan_destroy(None) == 0
    assert lib.gattn_plan_export(None, *([None] * 11)) == 1
    assert lib.gattn_plan_export_tiles(None, *([None] * 5)) == 1
    assert lib.gattn_plan_export_tile_bwd(None, *([None] * 7)) == 1
    assert b"plan is NULL" in lib.gattn_last_error()
    n = ctypes.c_size_t()
    assert lib.gattn_workspace_size(None, 2, 16, 0, ctypes.byref(n)) == 1
    assert lib.gattn_plan_set_wait_test(None, 1) == 1
    assert lib.gattn_plan_check_errors(None) == 1
    assert lib.gattn_fwd_noalloc(None, 2, 16, 0, None, None, None, None, None, None, None) == 1


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        gb.load_library(str(tmp_path / "nope.so"))


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "gnn_sparse_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, fn)) as f:
                    text = f.read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), fn
                assert "gattn_oracle" not in text, fn
