"""The C-ABI library loads and exports every symbol include/pkd.h declares."""
import ctypes
import os
import re

import paged_kv_decode_plan_gb300 as pkd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "pkd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkd_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(pkd.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = pkd.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version():
    assert pkd.abi_version() == 5 == pkd.ABI_VERSION


def test_struct_sizes_match_c_layout():
    # pkd_problem: 6 x int32, int64, 6 x int32 ; pkd_plan_t: problem + 4 x
    # int32 + 3 x int64 + 2 x int32
    assert ctypes.sizeof(pkd.Problem) == 56
    assert ctypes.sizeof(pkd.Plan) == 104
