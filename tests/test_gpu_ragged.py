"""GPU parity on shapes that are not multiples of 64 (zero-padded edge
GroupTiles): encode byte for byte against the oracle, products within the
bound (fp16) or exact (int8), Y written only inside [N][M]."""
import numpy as np
import pytest
import torch

import bitmap_encoded_unstructured_gb300 as bsp
import oracle
from bitmap_encoded_unstructured_gb300 import synth
from helpers import assert_within_bound, to_dev, to_dev_f16, tune

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture
def splitk(monkeypatch):
    def set_(s):
        if s is None:
            tune("splitk")
            tune("narrow_ctas")
        else:
            tune("splitk", str(s))
            tune("narrow_ctas", str(s))
    yield set_
    tune("splitk")
    tune("narrow_ctas")


def _encode(W):
    return bsp.BitmapMatrix(to_dev_f16(W, DEV) if W.dtype == np.uint16 else to_dev(W, DEV))


def _np(t):
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.float16 else a


F16_SHAPES = [(100, 72), (1, 8), (65, 136), (130, 200), (64, 1480), (330, 1480)]


@pytest.mark.parametrize("M,K", F16_SHAPES)
def test_encode_ragged_matches_oracle_bytes(M, K):
    W = synth.weights_f16(M, K, 0.5, "bernoulli", M * 7 + K)
    enc = oracle.encode(W)
    A = _encode(W)
    bm, off, vals = A.arrays()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bm.cpu().numpy().view(np.uint64), enc["bitmaps"])
    np.testing.assert_array_equal(off.cpu().numpy().view(np.uint32), enc["offsets"])
    np.testing.assert_array_equal(_np(vals), enc["values"])
    assert A.storage_bytes() == oracle.storage_bytes(enc)
    assert abs(A.cr() - oracle.compression_ratio(enc)) < 1e-12
    np.testing.assert_array_equal(_np(A.decode()), W)


@pytest.mark.parametrize("M,K", [(100, 208), (70, 144), (1, 16)])
def test_encode_ragged_int8(M, K):
    W = synth.weights_i8(M, K, 0.6, M + K)
    enc = oracle.encode(W)
    A = _encode(W)
    bm, off, vals = A.arrays()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bm.cpu().numpy().view(np.uint64), enc["bitmaps"])
    np.testing.assert_array_equal(vals.cpu().numpy(), enc["values"])
    np.testing.assert_array_equal(A.decode().cpu().numpy(), W)


@pytest.mark.parametrize("N", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("M,K", [(100, 200), (330, 1480), (65, 8)])
def test_spmm_ragged_decode_path(M, K, N, splitk):
    W = synth.weights_f16(M, K, 0.5, "uniform", M + 3 * K + N)
    X = synth.activations_f16(N, K, 11 * N + K)
    Yref, S = oracle.spmm_f16(W, X)
    A = _encode(W)
    for s in (1, 3, None):
        splitk(s)
        assert_within_bound(A.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, f"{M}x{K} N={N} splitk={s}")
    A.check()


@pytest.mark.parametrize("N", [17, 40, 300])
@pytest.mark.parametrize("M,K", [(200, 456), (130, 1000), (257, 72)])
def test_spmm_ragged_prefill(M, K, N):
    W = synth.weights_f16(M, K, 0.5, "uniform", 5 * M + K + N)
    X = synth.activations_f16(N, K, 13 * N + K)
    Yref, S = oracle.spmm_f16(W, X)
    A = _encode(W)
    assert_within_bound(A.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, f"prefill {M}x{K} N={N}")
    A.check()


@pytest.mark.parametrize("N", [1, 8, 16, 20])
def test_spmm_ragged_int8_exact(N, splitk):
    W = synth.weights_i8(100, 208, 0.5, 77 + N)
    X = synth.activations_i8(N, 208, 78 + N)
    A = _encode(W)
    for s in (1, 2, None):
        splitk(s)
        Y = A.spmm(to_dev(X, DEV)).cpu().numpy()
        np.testing.assert_array_equal(Y.astype(np.int64), oracle.spmm_i8(W, X))


@pytest.mark.parametrize("t", [None, 0.0, 0.5])
def test_spmspv_ragged(t):
    M, K = 150, 1480
    W = synth.weights_f16(M, K, 0.5, "uniform", 91)
    x = synth.activations_relu_f16(K, 92)
    A = _encode(W)
    if t is None:
        yref, s = oracle.spmspv_f16(W, x)
        y = A.spmspv(to_dev_f16(x, DEV))
    else:
        yref, s = oracle.spmspv_threshold_f16(W, x, t)
        y = A.spmspv_threshold(to_dev_f16(x, DEV), t)
    assert_within_bound(y.cpu().numpy().reshape(1, -1), yref.reshape(1, -1), s.reshape(1, -1), f"spmspv t={t}")
    A.check()


@pytest.mark.parametrize("N", [1, 5, 40])
def test_ragged_guard_bands(N):
    """Rows past M are padding: nothing is written outside Y [N][M]."""
    M, K = 100, 72
    W = synth.weights_f16(M, K, 0.5, "uniform", 23 + N)
    X = synth.activations_f16(N, K, 24 + N)
    A = _encode(W)
    pad = 256
    buf = torch.full((pad + N * M + pad,), 12345.0, dtype=torch.float16, device=DEV)
    Y = buf[pad:pad + N * M].view(N, M)
    A.spmm(to_dev_f16(X, DEV), out=Y)
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == np.float16(12345.0)) and np.all(b[-pad:] == np.float16(12345.0))
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y.cpu().numpy(), Yref, S, "ragged guard")


def test_import_ragged_oracle_encoding_and_padding_check():
    M, K = 100, 72
    W = synth.weights_f16(M, K, 0.5, "uniform", 31)
    X = synth.activations_f16(3, K, 32)
    enc = oracle.encode(W)
    B = bsp.BitmapMatrix.from_arrays(enc["bitmaps"], enc["offsets"], enc["values"], M, K)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(B.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, "imported ragged")
    # a bit set in the padding (row 100 of the padded grid) is rejected
    r, c = 100, 3
    g, p = oracle.locate(enc["Kp"], r, c)
    bm = enc["bitmaps"].copy()
    bm[g] |= np.uint64(1) << np.uint64(p)
    t = g // 64
    off = enc["offsets"].copy()
    off[t + 1:] += 1
    vals = np.concatenate([enc["values"][:off[t + 1] - 1], np.array([0x3C00], dtype=np.uint16),
                           enc["values"][off[t + 1] - 1:]])
    with pytest.raises(bsp.BspError) as e:
        bsp.BitmapMatrix.from_arrays(bm, off, vals, M, K)
    assert e.value.status == 1
