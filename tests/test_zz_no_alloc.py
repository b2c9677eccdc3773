"""bsp_spmm_noalloc: the decode-path product for callers that cannot allocate.

Some callers of this library may not call cudaMalloc (an operator that its
host framework hands only input and output buffers, a real-time loop, an
arena-managed process).  They keep the encoded arrays in their own memory
and call bsp_spmm_noalloc, which uses scratch compiled into the library.
These tests call it through the C ABI on arrays exported into caller-owned
buffers and hold its output against bsp_spmm's, on two calls in a row.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import bitmap_encoded_unstructured_gb300 as bsp
from bitmap_encoded_unstructured_gb300 import synth

from helpers import assert_within_bound, to_dev, to_dev_f16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _caller_arrays(A):
    """Copies of the encoded arrays in caller-owned buffers; the values
    buffer gets 16 bytes of readable slack past the last value."""
    o = bsp.bsp_info(A.h)
    dev = torch.device("cuda:0")
    bm = torch.empty(o.NBT, dtype=torch.int64, device=dev)
    off = torch.empty(o.NGT + 1, dtype=torch.int32, device=dev)
    esz = 2 if A.dtype == bsp.BSP_FP16 else 1
    vals = torch.zeros(o.NNZ * esz + 16, dtype=torch.uint8, device=dev)
    bsp.bsp_export(A.h, bm.data_ptr(), off.data_ptr(), vals.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return bm, off, vals


def _noalloc(A, arrays, X, N, Y):
    bm, off, vals = arrays
    L = bsp.lib()
    return L.bsp_spmm_noalloc(bm.data_ptr(), off.data_ptr(), vals.data_ptr(), A.dtype, A.M, A.K,
                              X.data_ptr(), N, Y.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("N", [1, 3, 5, 16])
def test_noalloc_matches_spmm_fp16(N):
    M, K = 384, 2048
    W = synth.weights_f16(M, K, 0.5, "uniform", 201)
    X = synth.activations_f16(N, K, 202)
    dev = torch.device("cuda:0")
    A = bsp.BitmapMatrix(to_dev_f16(W, dev))
    arrays = _caller_arrays(A)
    Xd = to_dev_f16(X, dev)
    ref = A.spmm(Xd).cpu().numpy()
    Yref, S = oracle.spmm_f16(W, X)
    for _ in range(2):  # two calls in a row share the scratch
        Y = torch.full((N, M), float("nan"), dtype=torch.float16, device=dev)
        assert _noalloc(A, arrays, Xd, N, Y) == 0
        got = Y.cpu().numpy()
        assert_within_bound(got, Yref, S, f"noalloc N={N}")
        # and against bsp_spmm: both are within the bound of the exact result
        diff = np.abs(got.astype(np.float64) - ref.astype(np.float64))
        assert np.all(diff <= 2 * (4e-3 * S + 1e-5))


def test_noalloc_matches_spmm_int8_exact():
    M, K = 256, 1024
    W = synth.weights_i8(M, K, 0.5, 211)
    X = synth.activations_i8(8, K, 212)
    dev = torch.device("cuda:0")
    A = bsp.BitmapMatrix(to_dev(W, dev))
    arrays = _caller_arrays(A)
    Xd = to_dev(X, dev)
    ref = A.spmm(Xd).cpu().numpy()
    for _ in range(2):
        Y = torch.zeros((8, M), dtype=torch.int32, device=dev)
        assert _noalloc(A, arrays, Xd, 8, Y) == 0
        np.testing.assert_array_equal(Y.cpu().numpy(), ref)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = bsp.lib()
    too_big = 32768 + 64  # BSP_NOALLOC_MAX_M + 64
    # rejected before any device work, so dummy aligned pointers suffice
    assert L.bsp_spmm_noalloc(256, 256, 256, 0, too_big, 64, 256, 1, 256, None) == 2
    assert L.bsp_spmm_noalloc(256, 256, 256, 0, 64, 64, 256, 17, 256, None) == 2
