"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Encode/decode and int8 are compared bit for bit; fp16 products within
|y - y_ref| <= 4e-3 * sum_k |w_mk x_kn| + 1e-5 per element; products whose
partial sums are small integers must be exact.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
import bitmap_encoded_unstructured_gb300 as bsp
from bitmap_encoded_unstructured_gb300 import synth

from helpers import assert_within_bound, sample_rows, to_dev, to_dev_f16, tune

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(autouse=True)
def _need_gpu():
    if DEV is None:
        pytest.skip("no CUDA device")


@pytest.fixture
def splitk(monkeypatch):
    """Force the split-K factor of the decode and narrow kernels for one test."""
    def set_(v):
        if v is None:
            tune("splitk")
            tune("narrow_ctas")
        else:
            tune("splitk", str(v))
            tune("narrow_ctas", str(v))
    yield set_
    tune("splitk")
    tune("narrow_ctas")


@pytest.fixture(params=["cuda_cores", "tcgen05_narrow"])
def path(request, monkeypatch):
    """fp16 N <= 16 on the CUDA-core decode kernels, or on the tcgen05
    narrow kernel (every N forced onto it)."""
    tune("narrow_min_n", "17" if request.param == "cuda_cores" else "1")
    yield request.param
    tune("narrow_min_n")


def _encode(W):
    if W.dtype == np.uint16:
        return bsp.BitmapMatrix(to_dev_f16(W, DEV))
    return bsp.BitmapMatrix(to_dev(W, DEV))


def _arrays_np(A):
    bm, off, vals = A.arrays()
    torch.cuda.synchronize()
    v = vals.cpu().numpy()
    v = v.view(np.uint16) if v.dtype == np.float16 else v
    return bm.cpu().numpy().view(np.uint64), off.cpu().numpy().view(np.uint32), v


# ------------------------------------------------------------------ format

ENC_CASES = [
    ("c1_256_bern50", lambda: synth.weights_f16(256, 256, 0.5, "bernoulli", synth.seed_for(1, 0))),
    ("sweep_30", lambda: synth.weights_f16(512, 1024, 0.3, "uniform", synth.seed_for(3, 0))),
    ("sweep_70", lambda: synth.weights_f16(512, 1024, 0.7, "uniform", synth.seed_for(3, 4))),
    ("magnitude_50", lambda: synth.weights_f16(384, 640, 0.5, "magnitude", synth.seed_for(2, 0))),
    ("int8_60", lambda: synth.weights_i8(256, 512, 0.6, synth.seed_for(5, 1))),
    ("all_zero", lambda: np.zeros((128, 192), dtype=np.uint16)),
    ("dense", lambda: synth.weights_f16(64, 128, 0.0, "none", 5)),
    ("single_nz", lambda: _single_nonzero()),
]


def _single_nonzero():
    W = np.zeros((192, 128), dtype=np.uint16)
    W[77, 99] = 0x3C00
    return W


@pytest.mark.parametrize("name,make", ENC_CASES, ids=[c[0] for c in ENC_CASES])
def test_encode_matches_oracle_bytes(name, make):
    W = make()
    enc = oracle.encode(W)
    A = _encode(W)
    bm, off, vals = _arrays_np(A)
    assert A.nnz == enc["NNZ"]
    np.testing.assert_array_equal(bm, enc["bitmaps"])
    np.testing.assert_array_equal(off, enc["offsets"])
    np.testing.assert_array_equal(vals, enc["values"])
    assert A.storage_bytes() == oracle.storage_bytes(enc)
    assert abs(A.cr() - oracle.compression_ratio(enc)) < 1e-12
    Wd = A.decode()
    torch.cuda.synchronize()
    got = Wd.cpu().numpy()
    got = got.view(np.uint16) if got.dtype == np.float16 else got
    np.testing.assert_array_equal(got, W)


def test_decode_special_payloads_bitwise():
    W = np.zeros((64, 128), dtype=np.uint16)
    for i, v in enumerate([0x8000, 0x7C00, 0xFC00, 0x7E00, 0x7C01, 0x0001, 0x8001]):
        W[5 * i, 3 * i + 2] = v
    A = _encode(W)
    assert A.nnz == 7
    got = A.decode().cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, W)


# ------------------------------------------------------------------ fp16 products

@pytest.mark.parametrize("N", [1, 8])
def test_spmm_tiny_config(N):
    """256x256 fp16, 50% Bernoulli zeros, X N(0,1)."""
    W = synth.weights_f16(256, 256, 0.5, "bernoulli", synth.seed_for(1, 0))
    X = synth.activations_f16(N, 256, synth.seed_for(1, 1))
    Y = _encode(W).spmm(to_dev_f16(X, DEV)).cpu().numpy()
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y, Yref, S, f"tiny N={N}")


@pytest.mark.parametrize("N", list(range(1, 17)))
def test_spmm_every_n_ragged(N, splitk, path):
    """Every N in 1..16 (padded register tiles), several tiles, odd split."""
    W = synth.weights_f16(384, 1472, 0.5, "uniform", 77)   # K/64 = 23 GT columns
    X = synth.activations_f16(N, 1472, 78 + N)
    Yref, S = oracle.spmm_f16(W, X)
    A = _encode(W)
    for s in (1, 3, None):
        splitk(s)
        Y = A.spmm(to_dev_f16(X, DEV)).cpu().numpy()
        assert_within_bound(Y, Yref, S, f"{path} N={N} splitk={s}")


@pytest.mark.parametrize("s", [0.3, 0.4, 0.5, 0.6, 0.7])
def test_spmm_sparsity_sweep_small(s, path):
    W = synth.weights_f16(512, 1024, s, "uniform", synth.seed_for(3, int(s * 10)))
    X = synth.activations_f16(16, 1024, 5)
    Yref, S = oracle.spmm_f16(W, X)
    for N in (1, 4, 8, 16):
        Y = _encode(W).spmm(to_dev_f16(X[:N].copy(), DEV)).cpu().numpy()
        assert_within_bound(Y, Yref[:N], S[:N], f"s={s} N={N}")


@pytest.mark.parametrize("N", [1, 3, 16])
def test_spmm_small_integers_exact(N, splitk, path):
    """|w|,|x| <= 8, K = 256: every partial sum is an exact integer, so the
    fp16 output has exactly one correct value, in any summation order."""
    W = synth.small_int_f16((320, 256), -8, 8, seed=41, sparsity=0.5)
    X = synth.small_int_f16((N, 256), -8, 8, seed=42)
    Yref, _ = oracle.spmm_f16(W, X)
    A = _encode(W)
    for s in (1, 2, 4):
        splitk(s)
        for _ in range(2):  # second call: workspace and counters were cleared
            Y = A.spmm(to_dev_f16(X, DEV)).cpu().numpy().astype(np.float64)
            np.testing.assert_array_equal(Y, Yref)


def test_spmm_permutation_exact():
    M = K = 256
    perm = synth.rng(5).permutation(K)
    W = np.zeros((M, K), dtype=np.uint16)
    W[np.arange(M), perm] = 0x3C00
    X = synth.activations_f16(8, K, 6)
    Y = _encode(W).spmm(to_dev_f16(X, DEV)).cpu().numpy()
    np.testing.assert_array_equal(Y.view(np.uint16), X[:, perm])


def test_spmm_all_zero_weight(path):
    W = np.zeros((128, 256), dtype=np.uint16)
    X = synth.activations_f16(4, 256, 1)
    Y = _encode(W).spmm(to_dev_f16(X, DEV)).cpu().numpy()
    assert np.all(Y == 0)


def test_spmm_dense_weight_vs_library():
    """s = 0 reduces to a dense GEMM: also hold it against torch.matmul in fp64 on CPU."""
    W = synth.weights_f16(256, 512, 0.0, "none", 9)
    X = synth.activations_f16(8, 512, 10)
    Y = _encode(W).spmm(to_dev_f16(X, DEV)).cpu().numpy()
    ref = (torch.from_numpy(X.view(np.float16)).double() @ torch.from_numpy(W.view(np.float16)).double().T).numpy()
    Yref, S = oracle.spmm_f16(W, X)
    np.testing.assert_allclose(Yref, ref, rtol=1e-12, atol=1e-12)
    assert_within_bound(Y, Yref, S, "dense")


def test_spmm_large_n_column_blocks():
    W = synth.weights_f16(256, 512, 0.5, "uniform", 19)
    X = synth.activations_f16(40, 512, 20)
    A = _encode(W)
    Y = A.spmm(to_dev_f16(X, DEV)).cpu().numpy()
    A.check()
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y, Yref, S, "N=40")


def test_spmm_guard_bands(path):
    """Canaries around Y are untouched; only Y[N][M] is written."""
    W = synth.weights_f16(192, 256, 0.5, "uniform", 23)
    X = synth.activations_f16(5, 256, 24)
    A = _encode(W)
    pad = 64
    buf = torch.full((pad + 5 * 192 + pad,), 12345.0, dtype=torch.float16, device=DEV)
    Y = buf[pad:pad + 5 * 192].view(5, 192)
    A.spmm(to_dev_f16(X, DEV), out=Y)
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == np.float16(12345.0)) and np.all(b[-pad:] == np.float16(12345.0))
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y.cpu().numpy(), Yref, S, "guard")


# ------------------------------------------------------------------ int8

@pytest.mark.parametrize("N", [1, 8, 16])
@pytest.mark.parametrize("s", [0.5, 0.6])
def test_spmm_int8_exact(N, s, splitk):
    W = synth.weights_i8(256, 1088, s, synth.seed_for(5, int(s * 10)))
    X = synth.activations_i8(N, 1088, synth.seed_for(5, 7))
    Yref = oracle.spmm_i8(W, X)
    A = _encode(W)
    for k in (1, 5, None):
        splitk(k)
        Y = A.spmm(to_dev(X, DEV)).cpu().numpy()
        assert Y.dtype == np.int32
        np.testing.assert_array_equal(Y.astype(np.int64), Yref)


@pytest.mark.parametrize("N", [1, 16])
def test_spmm_int8_scaled_bitexact(N):
    W = synth.weights_i8(192, 512, 0.5, synth.seed_for(5, 2))
    X = synth.activations_i8(N, 512, synth.seed_for(5, 3))
    scale = synth.row_scales(192, synth.seed_for(5, 4))
    ref = oracle.scale_i8(oracle.spmm_i8(W, X), scale)
    Y = _encode(W).spmm_scaled(to_dev(X, DEV), to_dev(scale, DEV)).cpu().numpy()
    np.testing.assert_array_equal(Y.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ spMspV

@pytest.mark.parametrize("zero_frac_shift", [None, -3.0, 0.5])
def test_spmspv_matches_n1_product(zero_frac_shift):
    M, K = 320, 2048
    W = synth.weights_f16(M, K, 0.5, "magnitude", synth.seed_for(2, 3))
    if zero_frac_shift is None:
        x = synth.activations_relu_f16(K, synth.seed_for(2, 4))
    else:
        x = synth.activations_relu_f16(K, 9, shift=zero_frac_shift)
    yref, s = oracle.spmspv_f16(W, x)
    A = _encode(W)
    y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
    assert_within_bound(y, yref, s, "spmspv")


def test_spmspv_all_zero_and_dense_x():
    M, K = 192, 1024
    W = synth.weights_f16(M, K, 0.5, "uniform", 31)
    A = _encode(W)
    y = A.spmspv(torch.zeros(K, dtype=torch.float16, device=DEV)).cpu().numpy()
    assert np.all(y == 0)
    x = synth.activations_f16(1, K, 32)[0]
    yref, s = oracle.spmspv_f16(W, x)
    assert_within_bound(A.spmspv(to_dev_f16(x, DEV)).cpu().numpy(), yref, s, "dense x")


def test_spmspv_small_integers_exact():
    W = synth.small_int_f16((256, 256), -8, 8, seed=51, sparsity=0.5)
    x = synth.small_int_f16((256,), 0, 8, seed=52, sparsity=0.8)
    yref, _ = oracle.spmspv_f16(W, x)
    y = _encode(W).spmspv(to_dev_f16(x, DEV)).cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(y, yref)


def test_spmspv_int8_exact():
    W = synth.weights_i8(256, 1024, 0.5, 61)
    x = synth.activations_i8(1, 1024, 62)[0]
    x[synth.rng(63).random(1024) < 0.85] = 0
    yref = oracle.spmm_i8(W, x.reshape(1, -1))[0]
    y = _encode(W).spmspv(to_dev(x, DEV)).cpu().numpy()
    np.testing.assert_array_equal(y.astype(np.int64), yref)


# ------------------------------------------------------------------ host-buffer API

def test_spmm_host_buffers():
    W = synth.weights_f16(256, 512, 0.5, "uniform", 71)
    X = synth.activations_f16(8, 512, 72)
    A = _encode(W)
    Xh = torch.from_numpy(X.view(np.float16)).pin_memory()
    Yh = torch.empty((8, 256), dtype=torch.float16).pin_memory()
    A.spmm_host(Xh, Yh)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Yh.numpy(), Yref, S, "host")


def test_spmm_host_async_enqueued_calls():
    """bsp_spmm_host_async on three handles (fp16 at two N, int8), enqueued
    back to back on one stream with a single synchronisation: every Y in
    host memory is right afterwards, and the same handle called twice in a
    row (staging buffers reused in stream order) gives both results."""
    s = torch.cuda.Stream()
    W1 = synth.weights_f16(384, 1024, 0.5, "uniform", 73)
    W2 = synth.weights_i8(256, 512, 0.5, 74)
    A1, A2 = _encode(W1), _encode(W2)
    Xa = synth.activations_f16(3, 1024, 75)
    Xb = synth.activations_f16(12, 1024, 76)
    X8 = synth.activations_i8(16, 512, 77)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    Xah, Xbh, X8h = pin(Xa.view(np.float16)), pin(Xb.view(np.float16)), pin(X8)
    Yah = torch.empty((3, 384), dtype=torch.float16).pin_memory()
    Ybh = torch.empty((12, 384), dtype=torch.float16).pin_memory()
    Y8h = torch.empty((16, 256), dtype=torch.int32).pin_memory()
    A1.spmm_host_async(Xah, Yah, stream=s)
    A1.spmm_host_async(Xbh, Ybh, stream=s)
    A2.spmm_host_async(X8h, Y8h, stream=s)
    s.synchronize()
    A1.check(s)
    A2.check(s)
    for X, Yh in ((Xa, Yah), (Xb, Ybh)):
        Yref, S = oracle.spmm_f16(W1, X)
        assert_within_bound(Yh.numpy(), Yref, S, "host async")
    np.testing.assert_array_equal(Y8h.numpy().astype(np.int64), oracle.spmm_i8(W2, X8))


# ------------------------------------------------------------------ ABI errors

def test_abi_error_paths():
    W = synth.weights_f16(128, 128, 0.5, "uniform", 81)
    Wd = to_dev_f16(W, DEV)
    L = bsp.lib()
    h = ctypes.c_void_p()
    assert L.bsp_encode(Wd.data_ptr(), 0, 128, 100, None, ctypes.byref(h)) == 2  # fp16: K % 8
    assert L.bsp_encode(Wd.data_ptr() + 2, 0, 64, 64, None, ctypes.byref(h)) == 4
    A = bsp.BitmapMatrix(Wd)
    X = torch.zeros((4, 128), dtype=torch.float16, device=DEV)
    Y = torch.zeros((4, 128), dtype=torch.float16, device=DEV)
    assert L.bsp_spmm(A.h, X.data_ptr(), 0, Y.data_ptr(), None) == 1
    assert L.bsp_spmm(A.h, X.data_ptr() + 2, 1, Y.data_ptr(), None) == 4
    assert L.bsp_spmm_scaled(A.h, X.data_ptr(), 1, Y.data_ptr(), Y.data_ptr(), None) == 3
    torch.cuda.synchronize()


# ------------------------------------------------------------------ full-size layers, sampled rows

OPT13B = {"qkv": (15360, 5120), "out": (5120, 5120), "fc1": (20480, 5120), "fc2": (5120, 20480)}


@pytest.mark.parametrize("layer", list(OPT13B))
def test_opt13b_layers_sampled_rows(layer):
    """Full OPT-13B-shaped layers at the benchmark's launch configuration;
    the oracle checks 4 sampled rows of every 64-row strip, all N."""
    M, K = OPT13B[layer]
    li = list(OPT13B).index(layer)
    W = synth.weights_f16(M, K, 0.5, "magnitude", synth.seed_for(2, li))
    X = synth.activations_f16(16, K, synth.seed_for(2, 5))
    A = _encode(W)
    rows = sample_rows(M, 4, seed=li)
    Yref, S = oracle.spmm_f16(W[rows], X)
    for N in (1, 2, 8, 16):
        Y = A.spmm(to_dev_f16(X[:N].copy(), DEV)).cpu().numpy()
        assert_within_bound(Y[:, rows], Yref[:N], S[:N], f"{layer} N={N}")
    if layer == "fc2":
        x = synth.activations_relu_f16(K, synth.seed_for(2, 6))
        yref, s = oracle.spmm_f16(W[rows], x.reshape(1, -1))
        y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
        assert_within_bound(y[rows], yref[0], s[0], "fc2 spmspv")


# ------------------------------------------------------------------ bounded waits

def test_check_ok_after_normal_calls():
    W = synth.weights_f16(128, 256, 0.5, "uniform", 91)
    A = _encode(W)
    A.spmm(to_dev_f16(synth.activations_f16(2, 256, 92), DEV))
    A.check()


@pytest.mark.parametrize("spmspv", [False, True])
def test_wait_that_runs_out_reports_timeout(spmspv):
    """In the test build of the library (libbsp_test.so) each warp's producer
    skips its first GT's copies (a barrier nothing completes); the
    consumers' bounded wait gives up, the kernel records BSP_ERR_TIMEOUT and
    returns; the context stays usable and the next call is correct."""
    W = synth.weights_f16(256, 1024, 0.5, "uniform", 93)
    X = synth.activations_f16(1, 1024, 94)
    with bsp.test_library() as T:
        A = _encode(W)
        Xd = to_dev_f16(X, DEV)
        try:
            assert T.bsp_testing_set_stall(1) == 0 and T.bsp_testing_set_spin_cap(2000) == 0
            if spmspv:
                A.spmspv(Xd[0].contiguous())
            else:
                A.spmm(Xd)
            with pytest.raises(bsp.BspError) as e:
                A.check()
            assert e.value.status == 7
        finally:
            T.bsp_testing_set_stall(0)
            T.bsp_testing_set_spin_cap(0)
        A.check()  # cleared
        Y = A.spmm(Xd).cpu().numpy()
        Yref, S = oracle.spmm_f16(W, X)
        assert_within_bound(Y, Yref, S, "after timeout")
        A.check()
        A.close()


def test_spmspv_mixed_selective_and_whole_fetch():
    """GTs whose x is mostly zero take the selective two-step fetch, busy
    ones the one-step fetch: alternate them along K."""
    M, K = 256, 64 * 24
    W = synth.weights_f16(M, K, 0.5, "uniform", 401)
    x = synth.activations_f16(1, K, 402)[0].copy()
    g = synth.rng(403)
    for gj in range(K // 64):
        seg = x[gj * 64:(gj + 1) * 64]
        if gj % 3 == 1:      # two active octets: selective
            keep = np.zeros(64, dtype=bool)
            keep[8 * g.integers(0, 8)] = True
            keep[8 * g.integers(0, 8) + 3] = True
            seg[~keep] = 0
        elif gj % 3 == 2:    # no active octet
            seg[:] = 0
    yref, s = oracle.spmspv_f16(W, x)
    A = _encode(W)
    for _ in range(2):
        y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
        assert_within_bound(y, yref, s, "mixed spmspv")
    A.check()


# ------------------------------------------------------------------ import of a cached encoding

def test_import_roundtrip_device_arrays():
    W = synth.weights_f16(256, 512, 0.5, "uniform", 501)
    X = synth.activations_f16(8, 512, 502)
    A = _encode(W)
    bm, off, vals = A.arrays()
    B = bsp.BitmapMatrix.from_arrays(bm, off, vals, 256, 512)
    Xd = to_dev_f16(X, DEV)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(B.spmm(Xd).cpu().numpy(), Yref, S, "imported")
    got = B.decode().cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(got, W)
    assert B.storage_bytes() == A.storage_bytes()


@pytest.mark.parametrize("dt", ["f16", "i8"])
def test_import_oracle_encoding_from_host(dt):
    """The CPU oracle's own encoding, imported from host memory, runs on the GPU."""
    if dt == "f16":
        W = synth.weights_f16(192, 320, 0.6, "uniform", 511)
        X = synth.activations_f16(5, 320, 512)
    else:
        W = synth.weights_i8(192, 320, 0.6, 513)
        X = synth.activations_i8(5, 320, 514)
    enc = oracle.encode(W)
    B = bsp.BitmapMatrix.from_arrays(enc["bitmaps"], enc["offsets"], enc["values"], 192, 320)
    if dt == "f16":
        Yref, S = oracle.spmm_f16(W, X)
        assert_within_bound(B.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, "oracle encoding")
    else:
        Y = B.spmm(to_dev(X, DEV)).cpu().numpy()
        np.testing.assert_array_equal(Y.astype(np.int64), oracle.spmm_i8(W, X))


def test_import_rejects_inconsistent_offsets():
    W = synth.weights_f16(128, 256, 0.5, "uniform", 521)
    enc = oracle.encode(W)
    off = enc["offsets"].copy()
    off[3] += 1  # no longer the prefix sum of the bitmaps
    with pytest.raises(bsp.BspError) as e:
        bsp.BitmapMatrix.from_arrays(enc["bitmaps"], off, enc["values"], 128, 256)
    assert e.value.status == 1
    bm = enc["bitmaps"].copy()
    bm[5] ^= np.uint64(1)  # one more or one fewer nonzero than the offsets say
    with pytest.raises(bsp.BspError):
        bsp.BitmapMatrix.from_arrays(bm, enc["offsets"], enc["values"], 128, 256)


# ------------------------------------------------------------------ spMspV with a threshold

@pytest.mark.parametrize("t", [0.0, 0.1, 0.5, 1.0, 2.0, 4.0])
def test_spmspv_threshold_fp16(t):
    """Magnitude pruning of x: from nearly all octets active (t = 0.1) to
    mostly-idle GroupTiles on the selective fetch (t = 2, 4)."""
    M, K = 256, 64 * 40
    W = synth.weights_f16(M, K, 0.5, "uniform", 601)
    x = synth.activations_f16(1, K, 602)[0]
    yref, s = oracle.spmspv_threshold_f16(W, x, t)
    A = _encode(W)
    for _ in range(2):
        y = A.spmspv_threshold(to_dev_f16(x, DEV), t).cpu().numpy()
        assert_within_bound(y, yref, s, f"threshold {t}")
    if t == 0.0:
        y0 = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
        assert_within_bound(y0, yref, s, "spmspv")
    A.check()


def test_spmspv_threshold_int8_exact():
    W = synth.weights_i8(192, 1024, 0.5, 611)
    x = synth.activations_i8(1, 1024, 612)[0]
    for t in (0.0, 60.0, 120.0):
        yref = oracle.spmm_i8(W, oracle.prune_activations_i8(x, t).reshape(1, -1))[0]
        y = _encode(W).spmspv_threshold(to_dev(x, DEV), t).cpu().numpy()
        np.testing.assert_array_equal(y.astype(np.int64), yref)


def test_spmspv_threshold_rejects_negative():
    A = _encode(synth.weights_f16(64, 64, 0.5, "uniform", 621))
    x = torch.zeros(64, dtype=torch.float16, device=DEV)
    with pytest.raises(bsp.BspError):
        A.spmspv_threshold(x, -1.0)
