"""CPU checks of the boundary: the shared library builds for sm_103a, loads
without a GPU, and exports every function include/per.h declares; the Python
binding names exactly those functions.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "per.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(per_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def built_lib():
    from cdf_scan_gb300 import _build
    return _build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("per_create", "per_destroy", "per_update", "per_build_cdf", "per_sample",
                     "per_is_weights", "per_total", "per_resample", "per_check"):
        assert required in names


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (per_[a-z0-9_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"


def test_library_loads_and_binding_covers_header(built_lib):
    lib = ctypes.CDLL(built_lib)
    for name in declared_functions():
        assert hasattr(lib, name)
    import cdf_scan_gb300
    assert sorted(cdf_scan_gb300.SIGNATURES) == declared_functions()
    # a pure host call: status names
    lib.per_status_str.restype = ctypes.c_char_p
    assert lib.per_status_str(0) == b"PER_OK"
    assert b"TIMEOUT" in lib.per_status_str(4)


def test_library_is_built_for_sm_103a_only(built_lib):
    from cdf_scan_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "cdf_scan_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("oracle)", ""), f"{f} mentions the oracle"
