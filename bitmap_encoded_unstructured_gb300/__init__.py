"""bitmap_encoded_unstructured_gb300: bitmap-encoded unstructured sparse matmul on GB300.

Thin Python binding over ``libbsp.so`` (the C ABI declared in
``include/bsp.h``).  Every step of the computation runs in the library's
CUDA kernels; this module only marshals arguments.  PyTorch supplies device
memory and streams.

Two layers:

* ``bsp_*`` functions with the C names, taking raw pointers / ints;
* ``BitmapMatrix``, a handle owner with tensor-level methods.

The library is loaded on first use; if it is missing or fails to load, the
call raises ``RuntimeError`` (there is no fallback of any kind).

``test_library()`` routes the calls made inside a ``with`` block to
``libbsp_test.so``, the test build, which alone exports the switches of
``include/bsp_testing.h``.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsp.so")
TEST_LIB_PATH = os.path.join(_HERE, "libbsp_test.so")

BSP_FP16 = 0
BSP_INT8 = 1
BSP_DECODE_MAX_N = 16

STATUS = {
    0: "BSP_OK", 1: "BSP_ERR_INVALID_ARG", 2: "BSP_ERR_SHAPE", 3: "BSP_ERR_DTYPE",
    4: "BSP_ERR_ALIGN", 5: "BSP_ERR_OOM", 6: "BSP_ERR_CUDA", 7: "BSP_ERR_TIMEOUT",
    8: "BSP_ERR_INTERNAL",
}

# Entry points declared in include/bsp.h: name -> (restype, argtypes).
_P = C.c_void_p
_I64 = C.c_int64
SIGNATURES = {
    "bsp_status_string": (C.c_char_p, [C.c_int]),
    "bsp_encode": (C.c_int, [_P, C.c_int, _I64, _I64, _P, C.POINTER(_P)]),
    "bsp_destroy": (C.c_int, [_P]),
    "bsp_spmm": (C.c_int, [_P, _P, _I64, _P, _P]),
    "bsp_spmm_scaled": (C.c_int, [_P, _P, _I64, _P, _P, _P]),
    "bsp_spmspv": (C.c_int, [_P, _P, _P, _P]),
    "bsp_spmspv_threshold": (C.c_int, [_P, _P, C.c_float, _P, _P]),
    "bsp_spmm_host": (C.c_int, [_P, _P, _I64, _P, _P]),
    "bsp_spmm_host_async": (C.c_int, [_P, _P, _I64, _P, _P]),
    "bsp_storage_bytes": (C.c_int, [_P, C.POINTER(C.c_uint64)]),
    "bsp_cr": (C.c_int, [_P, C.POINTER(C.c_double)]),
    "bsp_info": (C.c_int, [_P, _P]),
    "bsp_decode": (C.c_int, [_P, _P, _P]),
    "bsp_export": (C.c_int, [_P, _P, _P, _P, _P]),
    "bsp_check": (C.c_int, [_P, _P]),
    "bsp_import": (C.c_int, [_P, _P, _P, C.c_int, _I64, _I64, C.c_uint64, _P, C.POINTER(_P)]),
    "bsp_spmm_noalloc": (C.c_int, [_P, _P, _P, C.c_int, _I64, _I64, _P, _I64, _P, _P]),
    "bsp_set_deterministic": (C.c_int, [_P, C.c_int]),
    "bsp_set_tuning": (C.c_int, [C.c_int, _I64]),
    "bsp_build_column_index": (C.c_int, [_P, _P]),
    "bsp_column_index_bytes": (C.c_int, [_P, C.POINTER(C.c_uint64)]),
    "bsp_column_index_export": (C.c_int, [_P, _P, _P, _P, _P, _P]),
    "bsp_get_tuning": (C.c_int, [C.c_int, C.POINTER(_I64)]),
    "bsp_union_encode": (C.c_int, [_P, C.c_int, _I64, _I64, _P, C.POINTER(_P)]),
    "bsp_union_destroy": (C.c_int, [_P]),
    "bsp_union_spmm": (C.c_int, [_P, _P, _I64, _P, _P]),
    "bsp_union_storage_bytes": (C.c_int, [_P, C.POINTER(C.c_uint64)]),
    "bsp_union_info": (C.c_int, [_P, _P]),
    "bsp_union_export": (C.c_int, [_P, _P, _P, _P, _P]),
    "bsp_union_decode": (C.c_int, [_P, _P, _P]),
    "bsp_union_check": (C.c_int, [_P, _P]),
    "bsp_union_encode_reordered": (C.c_int, [_P, C.c_int, _I64, _I64, _P, C.POINTER(_P)]),
    "bsp_union_export_perms": (C.c_int, [_P, _P, _P]),
    "bsp_reorder_rows": (C.c_int, [_P, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _P, C.POINTER(_I64)]),
}

# Entry points of the test build only (include/bsp_testing.h).
TESTING_SIGNATURES = {
    "bsp_testing_set_stall": (C.c_int, [C.c_int]),
    "bsp_testing_set_spin_cap": (C.c_int, [C.c_uint32]),
}

# bsp_tune_t of include/bsp.h
TUNE = {"splitk": 0, "narrow_ctas": 1, "union_splitk": 2, "narrow_min_n": 3,
        "prefill_ksplit": 4, "prefill_cstages": 5, "narrow_min_n_i8": 6}


class bsp_info_t(C.Structure):
    _fields_ = [("M", C.c_int64), ("K", C.c_int64), ("dtype", C.c_int32),
                ("gt_m", C.c_int32), ("gt_k", C.c_int32), ("device", C.c_int32),
                ("NGT", C.c_int64), ("NBT", C.c_int64), ("NNZ", C.c_uint64),
                ("bitmaps", C.c_void_p), ("offsets", C.c_void_p), ("values", C.c_void_p)]


class bsp_union_info_t(C.Structure):
    _fields_ = [("M", C.c_int64), ("K", C.c_int64), ("bits", C.c_int32), ("lt", C.c_int32),
                ("areas_r", C.c_int32), ("areas_c", C.c_int32), ("device", C.c_int32),
                ("NLT", C.c_int64), ("nnz", C.c_uint64), ("total_values", C.c_uint64),
                ("value_bytes", C.c_uint64), ("masks", C.c_void_p), ("offsets", C.c_void_p),
                ("values", C.c_void_p), ("reordered", C.c_int32)]


class BspError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


_lib = None
_test_lib = None
_use_test = 0
_lock = threading.Lock()


def _load(path: str, sigs: dict) -> C.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing")
    L = C.CDLL(path)
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def testing_lib() -> C.CDLL:
    """Load libbsp_test.so, the test build (same kernels, plus the switches
    of include/bsp_testing.h)."""
    global _test_lib
    with _lock:
        if _test_lib is None:
            _test_lib = _load(TEST_LIB_PATH, {**SIGNATURES, **TESTING_SIGNATURES})
        return _test_lib


def lib() -> C.CDLL:
    """Load libbsp.so (built by ``build.build_library`` / ``__graft_entry__.build``);
    inside ``test_library()``, the test build instead."""
    global _lib
    if _use_test:
        return testing_lib()
    with _lock:
        if _lib is None:
            _lib = _load(LIB_PATH, SIGNATURES)
        return _lib


@contextlib.contextmanager
def test_library():
    """Route this module's calls to libbsp_test.so inside the block.  Handles
    made inside must be used and closed inside."""
    global _use_test
    L = testing_lib()
    _use_test += 1
    try:
        yield L
    finally:
        _use_test -= 1


def set_tuning(knob: str, value: int) -> None:
    """bsp_set_tuning by name (a key of ``TUNE``)."""
    _check("bsp_set_tuning", lib().bsp_set_tuning(TUNE[knob], int(value)))


def get_tuning(knob: str) -> int:
    v = C.c_int64()
    _check("bsp_get_tuning", lib().bsp_get_tuning(TUNE[knob], C.byref(v)))
    return v.value


@contextlib.contextmanager
def tuning(**knobs):
    """Set tuning knobs (``TUNE`` names) for the block, then restore them."""
    old = {k: get_tuning(k) for k in knobs}
    try:
        for k, v in knobs.items():
            set_tuning(k, v)
        yield
    finally:
        for k, v in old.items():
            set_tuning(k, v)


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise BspError(fn, st)


# ---------------------------------------------------------------- raw C names

def bsp_status_string(status: int) -> str:
    return lib().bsp_status_string(status).decode()


def bsp_encode(W_ptr: int, dtype: int, M: int, K: int, stream: int = 0) -> int:
    h = C.c_void_p()
    _check("bsp_encode", lib().bsp_encode(W_ptr, dtype, M, K, stream, C.byref(h)))
    return h.value


def bsp_destroy(h: int) -> None:
    _check("bsp_destroy", lib().bsp_destroy(h))


def bsp_spmm(h: int, X_ptr: int, N: int, Y_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmm", lib().bsp_spmm(h, X_ptr, N, Y_ptr, stream))


def bsp_spmm_scaled(h: int, X_ptr: int, N: int, scale_ptr: int, Y_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmm_scaled", lib().bsp_spmm_scaled(h, X_ptr, N, scale_ptr, Y_ptr, stream))


def bsp_spmspv(h: int, x_ptr: int, y_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmspv", lib().bsp_spmspv(h, x_ptr, y_ptr, stream))


def bsp_spmspv_threshold(h: int, x_ptr: int, threshold: float, y_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmspv_threshold", lib().bsp_spmspv_threshold(h, x_ptr, threshold, y_ptr, stream))


def bsp_spmm_host(h: int, X_host_ptr: int, N: int, Y_host_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmm_host", lib().bsp_spmm_host(h, X_host_ptr, N, Y_host_ptr, stream))


def bsp_spmm_host_async(h: int, X_host_ptr: int, N: int, Y_host_ptr: int, stream: int = 0) -> None:
    _check("bsp_spmm_host_async", lib().bsp_spmm_host_async(h, X_host_ptr, N, Y_host_ptr, stream))


def bsp_storage_bytes(h: int) -> int:
    v = C.c_uint64()
    _check("bsp_storage_bytes", lib().bsp_storage_bytes(h, C.byref(v)))
    return v.value


def bsp_cr(h: int) -> float:
    v = C.c_double()
    _check("bsp_cr", lib().bsp_cr(h, C.byref(v)))
    return v.value


def bsp_info(h: int) -> bsp_info_t:
    o = bsp_info_t()
    _check("bsp_info", lib().bsp_info(h, C.byref(o)))
    return o


def bsp_set_deterministic(h: int, on: bool) -> None:
    _check("bsp_set_deterministic", lib().bsp_set_deterministic(h, 1 if on else 0))


def bsp_decode(h: int, W_out_ptr: int, stream: int = 0) -> None:
    _check("bsp_decode", lib().bsp_decode(h, W_out_ptr, stream))


def bsp_export(h: int, bitmaps_ptr, offsets_ptr, values_ptr, stream: int = 0) -> None:
    _check("bsp_export", lib().bsp_export(h, bitmaps_ptr, offsets_ptr, values_ptr, stream))


def bsp_import(bitmaps_ptr: int, offsets_ptr: int, values_ptr, dtype: int, M: int, K: int, nnz: int,
               stream: int = 0) -> int:
    h = C.c_void_p()
    _check("bsp_import", lib().bsp_import(bitmaps_ptr, offsets_ptr, values_ptr, dtype, M, K, nnz, stream,
                                          C.byref(h)))
    return h.value


def bsp_check(h: int, stream: int = 0) -> None:
    _check("bsp_check", lib().bsp_check(h, stream))


def bsp_spmm_noalloc(bitmaps_ptr: int, offsets_ptr: int, values_ptr: int, dtype: int, M: int, K: int,
                     X_ptr: int, N: int, Y_ptr: int, stream: int = 0) -> None:
    """Decode-path product from caller-owned encoded arrays; allocates nothing
    (for callers that may not call cudaMalloc).  See include/bsp.h."""
    _check("bsp_spmm_noalloc", lib().bsp_spmm_noalloc(bitmaps_ptr, offsets_ptr, values_ptr, dtype, M, K,
                                                      X_ptr, N, Y_ptr, stream))


# ---------------------------------------------------------------- tensor layer

def bsp_union_encode(W_ptr: int, bits: int, M: int, K: int, stream: int = 0) -> int:
    h = C.c_void_p()
    _check("bsp_union_encode", lib().bsp_union_encode(W_ptr, bits, M, K, stream, C.byref(h)))
    return h.value


def bsp_union_encode_reordered(W_ptr: int, bits: int, M: int, K: int, stream: int = 0) -> int:
    h = C.c_void_p()
    _check("bsp_union_encode_reordered", lib().bsp_union_encode_reordered(W_ptr, bits, M, K, stream, C.byref(h)))
    return h.value


def bsp_union_export_perms(h: int, perms_ptr: int, stream: int = 0) -> None:
    _check("bsp_union_export_perms", lib().bsp_union_export_perms(h, perms_ptr, stream))


def bsp_reorder_rows(tile, RA: int, CA: int, exact: bool = True):
    """Host row reordering of one int8 tile [H][KL]: (perm int32 [H], cost)."""
    import numpy as np
    t = np.ascontiguousarray(tile, dtype=np.int8)
    H, KL = t.shape
    perm = np.zeros(H, dtype=np.int32)
    cost = C.c_int64()
    _check("bsp_reorder_rows", lib().bsp_reorder_rows(t.ctypes.data, H, KL, RA, CA, 1 if exact else 0,
                                                      perm.ctypes.data, C.byref(cost)))
    return perm, cost.value


def bsp_union_destroy(h: int) -> None:
    _check("bsp_union_destroy", lib().bsp_union_destroy(h))


def bsp_union_spmm(h: int, X_ptr: int, N: int, Y_ptr: int, stream: int = 0) -> None:
    _check("bsp_union_spmm", lib().bsp_union_spmm(h, X_ptr, N, Y_ptr, stream))


def bsp_union_storage_bytes(h: int) -> int:
    v = C.c_uint64()
    _check("bsp_union_storage_bytes", lib().bsp_union_storage_bytes(h, C.byref(v)))
    return v.value


def bsp_union_info(h: int) -> bsp_union_info_t:
    o = bsp_union_info_t()
    _check("bsp_union_info", lib().bsp_union_info(h, C.byref(o)))
    return o


def bsp_union_export(h: int, masks_ptr, offsets_ptr, values_ptr, stream: int = 0) -> None:
    _check("bsp_union_export", lib().bsp_union_export(h, masks_ptr, offsets_ptr, values_ptr, stream))


def bsp_union_decode(h: int, W_out_ptr: int, stream: int = 0) -> None:
    _check("bsp_union_decode", lib().bsp_union_decode(h, W_out_ptr, stream))


def bsp_union_check(h: int, stream: int = 0) -> None:
    _check("bsp_union_check", lib().bsp_union_check(h, stream))


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class BitmapMatrix:
    """An encoded weight W (M x K) living on one GPU.

    ``BitmapMatrix(W)`` encodes a CUDA tensor ``W`` (float16 or int8,
    row-major [M][K]; K a multiple of 8 for float16, 16 for int8; edge
    GroupTiles are zero-padded when M or K is not a multiple of 64).
    ``spmm(X)`` takes
    X [N][K] and returns Y [N][M] (= (W @ X.T).T, the [tokens, features]
    layout).
    """

    def __init__(self, W, stream=None):
        import torch
        if not W.is_cuda or W.dim() != 2:
            raise ValueError("W must be a 2-D CUDA tensor")
        if W.dtype == torch.float16:
            self.dtype = BSP_FP16
        elif W.dtype == torch.int8:
            self.dtype = BSP_INT8
        else:
            raise TypeError("W must be float16 or int8")
        W = W.contiguous()
        self.M, self.K = W.shape
        self.device = W.device
        self.torch_dtype = W.dtype
        self.h = bsp_encode(W.data_ptr(), self.dtype, self.M, self.K, _stream(stream))

    @classmethod
    def from_arrays(cls, bitmaps, offsets, values, M: int, K: int, device=None, stream=None):
        """A handle from encoded arrays (tensors on the GPU or the CPU, or numpy
        arrays): bitmaps int64/uint64 [M*K/64], offsets int32/uint32 [NGT+1],
        values fp16 (or uint16 bits) / int8 [NNZ]; M*K counted on the grid
        padded to multiples of 64.  Validated on the device."""
        import numpy as np
        import torch

        def ptr(a):
            if isinstance(a, np.ndarray):
                return np.ascontiguousarray(a).ctypes.data, a
            a = a.contiguous()
            return a.data_ptr(), a

        vals = values
        is_i8 = (vals.dtype == np.int8) if isinstance(vals, np.ndarray) else (vals.dtype == torch.int8)
        obj = cls.__new__(cls)
        obj.dtype = BSP_INT8 if is_i8 else BSP_FP16
        obj.M, obj.K = M, K
        obj.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        obj.torch_dtype = torch.int8 if is_i8 else torch.float16
        (pb, kb), (po, ko), (pv, kv) = ptr(bitmaps), ptr(offsets), ptr(vals)
        nnz = int(vals.shape[0])
        obj.h = bsp_import(pb, po, pv if nnz else None, obj.dtype, M, K, nnz, _stream(stream))
        del kb, ko, kv
        return obj

    def close(self):
        if getattr(self, "h", None):
            bsp_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- accounting
    def storage_bytes(self) -> int:
        return bsp_storage_bytes(self.h)

    def cr(self) -> float:
        return bsp_cr(self.h)

    def info(self) -> dict:
        o = bsp_info(self.h)
        return {f: getattr(o, f) for f, _ in bsp_info_t._fields_}

    @property
    def nnz(self) -> int:
        return int(bsp_info(self.h).NNZ)

    # -- arrays of the format (copies)
    def arrays(self, stream=None):
        """Copies of (bitmaps int64 [NBT], offsets int32 [NGT+1], values [NNZ])."""
        import torch
        o = bsp_info(self.h)
        dev = self.device
        bm = torch.empty(o.NBT, dtype=torch.int64, device=dev)
        off = torch.empty(o.NGT + 1, dtype=torch.int32, device=dev)
        vals = torch.empty(o.NNZ, dtype=self.torch_dtype, device=dev)
        bsp_export(self.h, bm.data_ptr(), off.data_ptr(), vals.data_ptr() if o.NNZ else None,
                   _stream(stream))
        return bm, off, vals

    def check(self, stream=None):
        """Synchronise and raise if a kernel on this handle gave up a wait."""
        bsp_check(self.h, _stream(stream))

    # -- Tiled-CBC column index (column-skipping spMspV)
    def build_column_index(self, stream=None):
        _check("bsp_build_column_index", lib().bsp_build_column_index(self.h, _stream(stream)))

    def column_index_bytes(self) -> int:
        v = C.c_uint64()
        _check("bsp_column_index_bytes", lib().bsp_column_index_bytes(self.h, C.byref(v)))
        return v.value

    def column_index_arrays(self, stream=None):
        """Copies of (TileOffset int32 [NGT+1], ColInfo int32 [NGT*64], bitmaps
        int64 [NGT*64*4], values [NNZ]) of the column index."""
        import torch
        tr = -(-self.M // 256)
        tc = -(-self.K // 64)
        ngt = tr * tc
        dev = self.device
        off = torch.empty(ngt + 1, dtype=torch.int32, device=dev)
        ci = torch.empty(ngt * 64, dtype=torch.int32, device=dev)
        bm = torch.empty(ngt * 64 * 4, dtype=torch.int64, device=dev)
        nnz = self.nnz
        vals = torch.empty(nnz, dtype=self.torch_dtype, device=dev)
        _check("bsp_column_index_export", lib().bsp_column_index_export(
            self.h, off.data_ptr(), ci.data_ptr(), bm.data_ptr(), vals.data_ptr() if nnz else None,
            _stream(stream)))
        return off, ci, bm, vals

    def set_deterministic(self, on: bool = True):
        """Split-K partial sums added in a fixed order (bit-identical fp16
        outputs from call to call) instead of by atomic adds."""
        bsp_set_deterministic(self.h, on)

    # -- compute
    def _out(self, N, out, dtype):
        import torch
        if out is None:
            out = torch.empty((N, self.M), dtype=dtype, device=self.device)
        return out

    def spmm(self, X, out=None, stream=None):
        import torch
        N = X.shape[0]
        ydt = torch.float16 if self.dtype == BSP_FP16 else torch.int32
        Y = self._out(N, out, ydt)
        bsp_spmm(self.h, X.data_ptr(), N, Y.data_ptr(), _stream(stream))
        return Y

    def spmm_scaled(self, X, row_scale, out=None, stream=None):
        import torch
        N = X.shape[0]
        Y = self._out(N, out, torch.float32)
        bsp_spmm_scaled(self.h, X.data_ptr(), N, row_scale.data_ptr(), Y.data_ptr(), _stream(stream))
        return Y

    def spmspv(self, x, out=None, stream=None):
        import torch
        ydt = torch.float16 if self.dtype == BSP_FP16 else torch.int32
        y = out if out is not None else torch.empty(self.M, dtype=ydt, device=self.device)
        bsp_spmspv(self.h, x.data_ptr(), y.data_ptr(), _stream(stream))
        return y

    def spmspv_threshold(self, x, threshold, out=None, stream=None):
        import torch
        ydt = torch.float16 if self.dtype == BSP_FP16 else torch.int32
        y = out if out is not None else torch.empty(self.M, dtype=ydt, device=self.device)
        bsp_spmspv_threshold(self.h, x.data_ptr(), float(threshold), y.data_ptr(), _stream(stream))
        return y

    def spmm_host(self, X_host, Y_host, stream=None):
        bsp_spmm_host(self.h, X_host.data_ptr(), X_host.shape[0], Y_host.data_ptr(), _stream(stream))
        return Y_host

    def spmm_host_async(self, X_host, Y_host, stream=None):
        """Enqueued only: Y_host is valid after `stream` is synchronised."""
        bsp_spmm_host_async(self.h, X_host.data_ptr(), X_host.shape[0], Y_host.data_ptr(), _stream(stream))
        return Y_host

    def decode(self, out=None, stream=None):
        import torch
        W = out if out is not None else torch.empty((self.M, self.K), dtype=self.torch_dtype,
                                                    device=self.device)
        bsp_decode(self.h, W.data_ptr(), _stream(stream))
        return W


class UnionMatrix:
    """An integer weight W (M x K) in the IE-BME union-bitmap format on one
    GPU: ``UnionMatrix(W, bits)`` encodes a CUDA int8 tensor whose values lie
    in the signed ``bits``-bit range (4 or 8); ``spmm`` multiplies by an int8
    activation block X [N][K] into int32 Y [N][M]."""

    def __init__(self, W, bits: int, stream=None, reorder: bool = False):
        import torch
        if W.dtype != torch.int8 or not W.is_cuda or W.dim() != 2:
            raise TypeError("W must be a 2-D int8 CUDA tensor")
        W = W.contiguous()
        self.M, self.K = int(W.shape[0]), int(W.shape[1])
        self.bits = int(bits)
        self.device = W.device
        enc = bsp_union_encode_reordered if reorder else bsp_union_encode
        self.h = enc(W.data_ptr(), self.bits, self.M, self.K, _stream(stream))

    def close(self):
        if getattr(self, "h", None):
            bsp_union_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def storage_bytes(self) -> int:
        return bsp_union_storage_bytes(self.h)

    def info(self) -> dict:
        o = bsp_union_info(self.h)
        return {f: getattr(o, f) for f, _ in bsp_union_info_t._fields_}

    def arrays(self, stream=None):
        """Copies of (masks int64 [NLT * 16], offsets int32 [NLT + 1], values uint8 [value_bytes])."""
        import torch
        o = bsp_union_info(self.h)
        masks = torch.empty(o.NLT * 16, dtype=torch.int64, device=self.device)
        offsets = torch.empty(o.NLT + 1, dtype=torch.int32, device=self.device)
        values = torch.empty(o.value_bytes, dtype=torch.uint8, device=self.device)
        bsp_union_export(self.h, masks.data_ptr(), offsets.data_ptr(), values.data_ptr() if o.value_bytes else None,
                         _stream(stream))
        return masks, offsets, values

    def decode(self, stream=None):
        import torch
        W = torch.empty((self.M, self.K), dtype=torch.int8, device=self.device)
        bsp_union_decode(self.h, W.data_ptr(), _stream(stream))
        return W

    def perms(self, stream=None):
        """Copy of the per-LT row permutations (uint8 [NLT, 64]) of a reordered encoding."""
        import torch
        o = bsp_union_info(self.h)
        p = torch.empty((o.NLT, 64), dtype=torch.uint8, device=self.device)
        bsp_union_export_perms(self.h, p.data_ptr(), _stream(stream))
        return p

    def check(self, stream=None):
        bsp_union_check(self.h, _stream(stream))

    def spmm(self, X, out=None, stream=None):
        import torch
        N = int(X.shape[0])
        Y = out if out is not None else torch.empty((N, self.M), dtype=torch.int32, device=self.device)
        bsp_union_spmm(self.h, X.data_ptr(), N, Y.data_ptr(), _stream(stream))
        return Y
