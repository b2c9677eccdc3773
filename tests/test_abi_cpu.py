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


# ---- argument validation that needs no device: every entry point rejects a
# null handle or pointer, a bad dtype, shape or alignment with the status the
# header documents, before any CUDA call

OK, INVALID, SHAPE, DTYPE, ALIGN = 0, 1, 2, 3, 4
NULL = None
MIS = 0x1001  # a misaligned address; never dereferenced before the alignment check


def _c(lib, name, *args):
    return getattr(lib, name)(*args)


def test_null_handles_are_rejected(lib):
    L = bsp.lib()
    u64, f32p = ctypes.c_uint64(), ctypes.c_double()
    info, uinfo = bsp.bsp_info_t(), bsp.bsp_union_info_t()
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.addressof(buf)
    calls = [
        ("bsp_destroy", NULL), ("bsp_check", NULL, NULL),
        ("bsp_spmm", NULL, p, 1, p, NULL), ("bsp_spmm_scaled", NULL, p, 1, p, p, NULL),
        ("bsp_spmspv", NULL, p, p, NULL), ("bsp_spmspv_threshold", NULL, p, ctypes.c_float(0.5), p, NULL),
        ("bsp_spmm_host", NULL, p, 1, p, NULL), ("bsp_spmm_host_async", NULL, p, 1, p, NULL),
        ("bsp_storage_bytes", NULL, ctypes.byref(u64)), ("bsp_cr", NULL, ctypes.byref(f32p)),
        ("bsp_info", NULL, ctypes.byref(info)), ("bsp_set_deterministic", NULL, 1),
        ("bsp_export", NULL, p, p, p, NULL), ("bsp_decode", NULL, p, NULL),
        ("bsp_build_column_index", NULL, NULL), ("bsp_column_index_bytes", NULL, ctypes.byref(u64)),
        ("bsp_column_index_export", NULL, p, p, p, p, NULL),
        ("bsp_union_destroy", NULL), ("bsp_union_check", NULL, NULL),
        ("bsp_union_spmm", NULL, p, 1, p, NULL), ("bsp_union_storage_bytes", NULL, ctypes.byref(u64)),
        ("bsp_union_info", NULL, ctypes.byref(uinfo)), ("bsp_union_export", NULL, p, p, p, NULL),
        ("bsp_union_export_perms", NULL, p, NULL), ("bsp_union_decode", NULL, p, NULL),
    ]
    for name, *args in calls:
        assert getattr(L, name)(*args) == INVALID, name


def test_encode_and_import_validate_before_the_device(lib):
    L = bsp.lib()
    h = ctypes.c_void_p()
    out = ctypes.byref(h)
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16  # 16-B aligned inside buf
    assert L.bsp_encode(p, bsp.BSP_FP16, 64, 64, NULL, NULL) == INVALID           # no out
    assert L.bsp_encode(NULL, bsp.BSP_FP16, 64, 64, NULL, out) == INVALID
    assert L.bsp_encode(p, 7, 64, 64, NULL, out) == DTYPE
    assert L.bsp_encode(p, bsp.BSP_FP16, 0, 64, NULL, out) == SHAPE
    assert L.bsp_encode(p, bsp.BSP_FP16, 64, 12, NULL, out) == SHAPE               # K % 8
    assert L.bsp_encode(p, bsp.BSP_INT8, 64, 24, NULL, out) == SHAPE               # K % 16
    assert L.bsp_encode(MIS, bsp.BSP_FP16, 64, 64, NULL, out) == ALIGN
    assert h.value is None
    assert L.bsp_import(NULL, p, p, bsp.BSP_FP16, 64, 64, 1, NULL, out) == INVALID
    assert L.bsp_import(p, p, p, 7, 64, 64, 1, NULL, out) == DTYPE
    assert L.bsp_union_encode(NULL, 8, 64, 64, NULL, out) == INVALID
    assert L.bsp_union_encode(p, 5, 64, 64, NULL, out) == INVALID                  # bits 4 or 8
    assert L.bsp_union_encode(p, 8, 64, 24, NULL, out) == SHAPE                    # K % 16
    assert L.bsp_union_encode(p, 4, 64, 1 << 21, NULL, out) == SHAPE               # W4A4 exactness bound
    assert L.bsp_union_encode(MIS, 8, 64, 64, NULL, out) == ALIGN
    assert L.bsp_union_encode_reordered(NULL, 4, 64, 64, NULL, out) == INVALID


def test_noalloc_validates_before_the_device(lib):
    L = bsp.lib()
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    args = lambda **kw: [kw.get(k, v) for k, v in  # noqa: E731
                         (("bm", p), ("off", p), ("vals", p), ("dt", bsp.BSP_FP16), ("M", 64), ("K", 64),
                          ("X", p), ("N", 8), ("Y", p))] + [NULL]
    assert L.bsp_spmm_noalloc(*args(bm=NULL)) == INVALID
    assert L.bsp_spmm_noalloc(*args(Y=NULL)) == INVALID
    assert L.bsp_spmm_noalloc(*args(dt=7)) == DTYPE
    assert L.bsp_spmm_noalloc(*args(M=100)) == SHAPE          # multiples of 64 only
    assert L.bsp_spmm_noalloc(*args(N=0)) == SHAPE
    assert L.bsp_spmm_noalloc(*args(N=17)) == SHAPE           # the fixed scratch holds N <= 16
    assert L.bsp_spmm_noalloc(*args(M=64 * 1024)) == SHAPE    # and M <= 32768
    assert L.bsp_spmm_noalloc(*args(X=MIS)) == ALIGN
    assert L.bsp_spmm_noalloc(*args(off=p + 2)) == ALIGN      # offsets 4-B aligned


def test_reorder_rows_validates_its_tile(lib):
    L = bsp.lib()
    tile = (ctypes.c_int8 * 64)()
    perm = (ctypes.c_int32 * 8)()
    cost = ctypes.c_int64()
    assert L.bsp_reorder_rows(NULL, 8, 8, 2, 1, 1, perm, ctypes.byref(cost)) == INVALID
    assert L.bsp_reorder_rows(tile, 7, 8, 2, 1, 1, perm, ctypes.byref(cost)) == SHAPE   # H % RA
    assert L.bsp_reorder_rows(tile, 8, 8, 3, 1, 0, perm, ctypes.byref(cost)) == SHAPE   # heuristic: RA = 2
