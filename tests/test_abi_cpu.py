"""The C-ABI library builds, loads and exports every symbol include/*.h declares.

No compute call is made (there may be no GPU here).
"""
import ctypes
import glob
import os
import re

import pytest

import bitmap_encoded_unstructured_gb300 as bsp
from bitmap_encoded_unstructured_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


TESTING_HEADER = "bsp_testing.h"  # declared for the test build only


def _declared(testing=False):
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        if (os.path.basename(h) == TESTING_HEADER) != testing:
            continue
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(bsp_[a-z0-9_]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    build_library()
    return ctypes.CDLL(bsp.LIB_PATH)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "bsp_encode" in names and "bsp_spmm" in names and "bsp_spmspv" in names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_covers_every_symbol():
    assert _declared() == set(bsp.SIGNATURES)
    assert _declared(testing=True) == set(bsp.TESTING_SIGNATURES)


def test_testing_switches_only_in_the_test_build(lib):
    """The production library cannot be told to skip its copies or shorten
    its waits: those switches exist only in libbsp_test.so, which also
    exports everything the production library does."""
    t = ctypes.CDLL(bsp.TEST_LIB_PATH)
    for n in sorted(_declared(testing=True)):
        assert not hasattr(lib, n), f"{n} exported by the production library"
        assert hasattr(t, n), f"{n} missing from the test library"
    for n in sorted(_declared()):
        assert hasattr(t, n), f"{n} missing from the test library"


def test_tuning_knobs_without_gpu():
    """bsp_set_tuning / bsp_get_tuning round-trip and range checks (no GPU)."""
    L = bsp.lib()
    v = ctypes.c_int64()
    old = {}
    for name, k in bsp.TUNE.items():
        assert L.bsp_get_tuning(k, ctypes.byref(v)) == 0
        old[k] = v.value
    try:
        assert L.bsp_set_tuning(bsp.TUNE["splitk"], 7) == 0
        assert L.bsp_get_tuning(bsp.TUNE["splitk"], ctypes.byref(v)) == 0 and v.value == 7
        assert L.bsp_set_tuning(bsp.TUNE["splitk"], -1) == 1          # split counts >= 0
        assert L.bsp_set_tuning(bsp.TUNE["prefill_ksplit"], 2) == 1   # -1, 0 or 1
        assert L.bsp_set_tuning(bsp.TUNE["narrow_min_n"], 0) == 1     # >= 1
        assert L.bsp_set_tuning(99, 0) == 1                           # unknown knob
        assert L.bsp_get_tuning(bsp.TUNE["splitk"], None) == 1
    finally:
        for k, val in old.items():
            L.bsp_set_tuning(k, val)


def test_status_strings_without_gpu():
    for s in range(9):
        assert bsp.bsp_status_string(s)
    assert bsp.bsp_status_string(0) == "ok"


def test_argument_errors_without_gpu():
    # Calls rejected before any CUDA work return their status codes.
    L = bsp.lib()
    h = ctypes.c_void_p()
    assert L.bsp_encode(None, 0, 64, 64, None, ctypes.byref(h)) == 1   # null W
    assert L.bsp_encode(16, 0, 0, 64, None, ctypes.byref(h)) == 2      # M < 1
    assert L.bsp_encode(16, 0, 64, 60, None, ctypes.byref(h)) == 2     # fp16: K % 8
    assert L.bsp_encode(16, 1, 64, 72, None, ctypes.byref(h)) == 2     # int8: K % 16
    assert L.bsp_encode(16, 7, 64, 64, None, ctypes.byref(h)) == 3     # dtype
    assert L.bsp_encode(8, 0, 64, 64, None, ctypes.byref(h)) == 4      # alignment
    assert L.bsp_spmm(None, 16, 1, 16, None) == 1
    assert L.bsp_spmspv(None, 16, 16, None) == 1
    assert L.bsp_destroy(None) == 1
    assert L.bsp_set_deterministic(None, 1) == 1
    v = ctypes.c_uint64()
    assert L.bsp_storage_bytes(None, ctypes.byref(v)) == 1
