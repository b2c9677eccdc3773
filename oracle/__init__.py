"""CPU oracle for the bitmap-encoded unstructured sparse matmul.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this package; the CUDA library never imports it and the
two share no code.  The arithmetic lives in ``bsp_oracle.c`` (plain loops,
fp64 / int64); this module only builds it with gcc, loads it with ctypes and
marshals numpy arrays.

Accounting helpers (bytes of the oracle's own arrays, compression ratio,
CSR comparator, payload-to-metadata ratio) are computed from the arrays the
oracle actually produced, so that tests can hold them against the closed
forms printed on the pages.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``bsp_oracle.c`` into ``liboracle.so`` (gcc -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = C.CDLL(_LIB_PATH)
        p = C.c_void_p
        i64 = C.c_int64
        lib.oracle_half_to_double.argtypes = [C.c_uint16]
        lib.oracle_half_to_double.restype = C.c_double
        lib.oracle_popcount64.argtypes = [C.c_uint64]
        lib.oracle_popcount64.restype = C.c_int
        lib.oracle_rank.argtypes = [C.c_uint64, C.c_int]
        lib.oracle_rank.restype = C.c_int
        lib.oracle_locate.argtypes = [i64, i64, i64, C.POINTER(i64), C.POINTER(C.c_int)]
        lib.oracle_locate.restype = None
        lib.oracle_position.argtypes = [i64, i64, C.c_int, C.POINTER(i64), C.POINTER(i64)]
        lib.oracle_position.restype = None
        lib.oracle_encode_bitmaps.argtypes = [p, C.c_int, i64, i64, p]
        lib.oracle_encode_bitmaps.restype = C.c_uint64
        lib.oracle_encode_values.argtypes = [p, C.c_int, i64, i64, p, p, p]
        lib.oracle_encode_values.restype = None
        lib.oracle_decode.argtypes = [p, p, p, C.c_int, i64, i64, p]
        lib.oracle_decode.restype = None
        lib.oracle_spmm_f16.argtypes = [p, p, i64, i64, i64, p, p]
        lib.oracle_spmm_f16.restype = None
        lib.oracle_spmm_i8.argtypes = [p, p, i64, i64, i64, p]
        lib.oracle_spmm_i8.restype = None
        lib.oracle_scale_i8.argtypes = [p, p, i64, i64, p]
        lib.oracle_scale_i8.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = C.c_int
        lib.oracle_set_threads.argtypes = [C.c_int]
        lib.oracle_set_threads.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _elem_bytes(W: np.ndarray) -> int:
    if W.dtype == np.uint16:
        return 2
    if W.dtype == np.int8:
        return 1
    raise TypeError("W must be uint16 (fp16 bits) or int8")


# ---------------------------------------------------------------- scalars

def half_to_double(h: int) -> float:
    return _load().oracle_half_to_double(h)


def popcount64(x: int) -> int:
    return _load().oracle_popcount64(x)


def rank(bitmap: int, p: int) -> int:
    return _load().oracle_rank(bitmap, p)


def locate(K: int, r: int, c: int):
    g = C.c_int64()
    p = C.c_int()
    _load().oracle_locate(K, r, c, C.byref(g), C.byref(p))
    return g.value, p.value


def position(K: int, g: int, p: int):
    r = C.c_int64()
    c = C.c_int64()
    _load().oracle_position(K, g, p, C.byref(r), C.byref(c))
    return r.value, c.value


# ---------------------------------------------------------------- format

def _padded(n: int) -> int:
    return (n + 63) // 64 * 64


def encode(W: np.ndarray) -> dict:
    """Encode dense ``W`` (uint16 fp16 bits or int8, [M][K]) into the format.

    When M or K is not a multiple of 64 the grid of GroupTiles covers W
    padded with zeros to multiples of 64 (the edge GroupTiles are zero-padded;
    padding stores no values and its bits are 0).
    """
    W = np.ascontiguousarray(W)
    M, K = W.shape
    if M < 1 or K < 1:
        raise ValueError("M and K must be positive")
    Mp, Kp = _padded(M), _padded(K)
    if (Mp, Kp) != (M, K):
        Wp = np.zeros((Mp, Kp), dtype=W.dtype)
        Wp[:M, :K] = W
    else:
        Wp = W
    eb = _elem_bytes(W)
    lib = _load()
    NBT = Mp * Kp // 64
    NGT = (Mp // 64) * (Kp // 64)
    bitmaps = np.zeros(NBT, dtype=np.uint64)
    nnz = lib.oracle_encode_bitmaps(_ptr(Wp), eb, Mp, Kp, _ptr(bitmaps))
    offsets = np.zeros(NGT + 1, dtype=np.uint32)
    values = np.zeros(nnz, dtype=W.dtype)
    lib.oracle_encode_values(_ptr(Wp), eb, Mp, Kp, _ptr(bitmaps), _ptr(offsets),
                             _ptr(values) if nnz else None)
    return {"M": M, "K": K, "Mp": Mp, "Kp": Kp, "dtype": W.dtype, "NGT": NGT,
            "NBT": NBT, "NNZ": int(nnz), "bitmaps": bitmaps, "offsets": offsets,
            "values": values}


def decode(enc: dict) -> np.ndarray:
    M, K = enc["M"], enc["K"]
    Mp, Kp = enc.get("Mp", M), enc.get("Kp", K)
    out = np.empty((Mp, Kp), dtype=enc["dtype"])
    eb = 2 if enc["dtype"] == np.uint16 else 1
    vals = enc["values"]
    _load().oracle_decode(_ptr(enc["bitmaps"]), _ptr(enc["offsets"]),
                          _ptr(vals) if vals.size else None, eb, Mp, Kp, _ptr(out))
    return np.ascontiguousarray(out[:M, :K])


def storage_bytes(enc: dict) -> int:
    """Bytes the oracle's three arrays actually occupy (no padding)."""
    return int(enc["bitmaps"].nbytes + enc["offsets"].nbytes + enc["values"].nbytes)


def compression_ratio(enc: dict) -> float:
    """Same-dtype dense bytes over stored bytes."""
    vb = enc["values"].itemsize
    return vb * enc["M"] * enc["K"] / storage_bytes(enc)


def csr_bytes(W: np.ndarray) -> int:
    """Bytes of a CSR built the way the SpInfer page describes it: the
    nonzero values plus one 32-bit column index each, plus M+1 row pointers
    of 32 bits."""
    W = np.ascontiguousarray(W)
    nz = W != 0
    colidx = np.nonzero(nz)[1].astype(np.uint32)
    vals = W[nz]
    rowptr = np.zeros(W.shape[0] + 1, dtype=np.uint32)
    return int(vals.nbytes + colidx.nbytes + rowptr.nbytes)


def payload_to_metadata(enc: dict) -> float:
    """PMR = value bytes / index bytes (bitmaps + offsets)."""
    meta = enc["bitmaps"].nbytes + enc["offsets"].nbytes
    return enc["values"].nbytes / meta


# ---------------------------------------------------------------- product

def spmm_f16(W: np.ndarray, X: np.ndarray):
    """fp64 dense product of fp16 bits: returns (Y[N][M], sumabs[N][M])."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    X = np.ascontiguousarray(X, dtype=np.uint16)
    M, K = W.shape
    N, K2 = X.shape
    assert K == K2
    Y = np.empty((N, M), dtype=np.float64)
    S = np.empty((N, M), dtype=np.float64)
    _load().oracle_spmm_f16(_ptr(W), _ptr(X), M, K, N, _ptr(Y), _ptr(S))
    return Y, S


def spmm_i8(W: np.ndarray, X: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.int8)
    X = np.ascontiguousarray(X, dtype=np.int8)
    M, K = W.shape
    N, K2 = X.shape
    assert K == K2
    Y = np.empty((N, M), dtype=np.int64)
    _load().oracle_spmm_i8(_ptr(W), _ptr(X), M, K, N, _ptr(Y))
    return Y


def scale_i8(acc: np.ndarray, scale: np.ndarray) -> np.ndarray:
    acc = np.ascontiguousarray(acc, dtype=np.int64)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    N, M = acc.shape
    out = np.empty((N, M), dtype=np.float32)
    _load().oracle_scale_i8(_ptr(acc), _ptr(scale), M, N, _ptr(out))
    return out


def spmspv_f16(W: np.ndarray, x: np.ndarray):
    """The sparse-vector product is the N = 1 product: skipping x_k == 0
    removes only terms that are exactly zero."""
    Y, S = spmm_f16(W, np.ascontiguousarray(x, dtype=np.uint16).reshape(1, -1))
    return Y[0], S[0]


def prune_activations_f16(x: np.ndarray, threshold: float) -> np.ndarray:
    """Dynamic pruning by magnitude: x_k -> 0 where |x_k| <= threshold (the
    activation-magnitude criterion of SPDP's dynamic pruning).  fp16 bits in,
    fp16 bits out; the comparison is on the exact value (fp64); NaN is kept."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    t = np.float64(np.float32(threshold))
    v = np.array([half_to_double(int(b)) for b in x.reshape(-1)]).reshape(x.shape)
    out = x.copy()
    out[np.abs(v) <= t] = 0
    return out


def prune_activations_i8(x: np.ndarray, threshold: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.int8)
    t = np.float64(np.float32(threshold))
    out = x.copy()
    out[np.abs(x.astype(np.float64)) <= t] = 0
    return out


def spmspv_threshold_f16(W: np.ndarray, x: np.ndarray, threshold: float):
    """y = W * x' with x' the magnitude-pruned activations."""
    return spmspv_f16(W, prune_activations_f16(x, threshold))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(n)
