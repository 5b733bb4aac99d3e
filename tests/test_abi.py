"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/bh.h declares; the binding's constants match
the header; argument validation fails cleanly without a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bh.h")


def _header_functions():
    text = open(HEADER).read()
    return set(re.findall(r"^\s*(?:int|const char \*)\s*(bh_\w+)\s*\(", text, re.M))


def _header_defines():
    text = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(BH_\w+)\s+(\d+)\b", text)}


@pytest.fixture(scope="module")
def bhmod():
    import barnes_hut_body_gb300 as B
    if not os.path.exists(B.LIB_PATH):
        from barnes_hut_body_gb300 import build
        build.build()
    return B


def test_header_declares_the_abi():
    fns = _header_functions()
    for name in ("bh_create", "bh_set_params", "bh_compute", "bh_destroy",
                 "bh_direct", "bh_sync_status", "bh_compute_host"):
        assert name in fns


def test_library_exports_every_declared_symbol(bhmod):
    L = ctypes.CDLL(bhmod.LIB_PATH)
    for name in _header_functions():
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", bhmod.LIB_PATH],
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(bh_\w+)", out))
    assert _header_functions() <= exported
    assert set(bhmod.EXPORTED) == _header_functions()


def test_binding_constants_match_header(bhmod):
    for name, value in _header_defines().items():
        if hasattr(bhmod, name):
            assert getattr(bhmod, name) == value, name


def test_calls_without_a_device_fail_cleanly(bhmod):
    L = bhmod.lib()
    h = ctypes.c_void_p()
    rc = L.bh_create(ctypes.byref(h), 9999, 0, 0)
    assert rc == bhmod.BH_EINVAL and not h.value
    assert L.bh_set_params(None, 0.5, 1.0, 0.0) == bhmod.BH_EINVAL
    assert L.bh_compute(None, None, 0, None, 0, None, None) == bhmod.BH_EINVAL
    assert L.bh_destroy(None) == bhmod.BH_OK
    assert L.bh_last_error(None) == b"null context"
    assert L.bh_neighbors(None, None, None, 0, 2.0, 1, None, None, None, 0, None) == bhmod.BH_EINVAL
    assert L.bh_leapfrog(None, None, None, 0, None, 1e-3, 1, 0, None) == bhmod.BH_EINVAL
    assert L.bh_set_option(None, bhmod.BH_OPT_ESTIMATOR, 1) == bhmod.BH_EINVAL
    assert L.bh_fp32_probe(None, 0, 1, None, None) == bhmod.BH_EINVAL


def test_product_path_does_not_import_the_oracle():
    """The library package must not reach the CPU oracle."""
    pkg = os.path.join(ROOT, "barnes_hut_body_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "bh_oracle" not in text, f
