"""GPU parity of the IE-BME union-bitmap format and its product (W8A8,
W4A4) against the oracle: the encoded arrays byte for byte, the round trip,
the storage bytes, and exact int32 products."""
import numpy as np
import pytest
import torch

import bitmap_encoded_unstructured_gb300 as bsp
from oracle import ie_bme as u
from helpers import sample_rows, tune

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _weights(M, K, bits, s, seed):
    rng = np.random.default_rng(seed)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1))
    W = rng.integers(lo, hi, size=(M, K)) * (rng.random((M, K)) >= s)
    return W.astype(np.int8)


def _acts(N, K, bits, seed):
    rng = np.random.default_rng(seed)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1))
    return rng.integers(lo, hi, size=(N, K)).astype(np.int8)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,s", [(64, 64, 0.5), (130, 208, 0.6), (1, 16, 0.0), (256, 512, 0.9), (192, 320, 1.0)])
def test_encode_matches_oracle_bytes(M, K, s, bits):
    W = _weights(M, K, bits, s, 10 * M + K + bits)
    enc = u.union_encode(W, bits)
    A = bsp.UnionMatrix(_dev(W), bits)
    masks, offsets, values = A.arrays()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(masks.cpu().numpy().view(np.uint64), enc["masks"])
    np.testing.assert_array_equal(offsets.cpu().numpy().view(np.uint32), enc["offsets"])
    np.testing.assert_array_equal(values.cpu().numpy(), u.pack_values(enc["values"], bits))
    assert A.storage_bytes() == u.storage_bytes(enc)
    info = A.info()
    assert info["nnz"] == enc["nnz"] and info["total_values"] == int(enc["offsets"][-1])
    np.testing.assert_array_equal(A.decode().cpu().numpy(), W)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N", [1, 2, 3, 8, 13, 16, 20])
@pytest.mark.parametrize("M,K", [(256, 1024), (130, 208)])
def test_spmm_exact(M, K, N, bits):
    W = _weights(M, K, bits, 0.5, M + K + N + bits)
    X = _acts(N, K, bits, 7 * N + bits)
    A = bsp.UnionMatrix(_dev(W), bits)
    Y = A.spmm(_dev(X)).cpu().numpy().astype(np.int64)
    A.check()
    np.testing.assert_array_equal(Y, u.union_spmm(W, X))


@pytest.mark.parametrize("splits", [1, 3, 16])
def test_spmm_split_k_forced(splits, monkeypatch):
    """Every split count gives the same exact result, call after call (the
    workspace and counters are clean after each)."""
    W = _weights(320, 1024, 4, 0.6, 41)
    X = _acts(8, 1024, 4, 42)
    ref = u.union_spmm(W, X)
    tune("union_splitk", str(splits))
    A = bsp.UnionMatrix(_dev(W), 4)
    Xd = _dev(X)
    for _ in range(3):
        np.testing.assert_array_equal(A.spmm(Xd).cpu().numpy().astype(np.int64), ref)
    A.check()


def test_spmm_extremes_int8():
    """Full-range int8 weights and activations, dense: exact int32."""
    W = np.full((128, 4096), -128, dtype=np.int8)
    X = np.full((2, 4096), -128, dtype=np.int8)
    A = bsp.UnionMatrix(_dev(W), 8)
    Y = A.spmm(_dev(X)).cpu().numpy().astype(np.int64)
    assert np.all(Y == 128 * 128 * 4096)


@pytest.mark.parametrize("w,x", [(-8, -8), (7, -8), (-8, 7)])
def test_spmm_extremes_int4(w, x):
    """Dense int4 extremes, N = 3: exact int32 (the int4 path accumulates
    16 w x per product and divides by 16 after the reduction)."""
    K = 8192
    W = np.full((192, K), w, dtype=np.int8)
    X = np.full((3, K), x, dtype=np.int8)
    A = bsp.UnionMatrix(_dev(W), 4)
    Y = A.spmm(_dev(X)).cpu().numpy().astype(np.int64)
    A.check()
    assert np.all(Y == w * x * K)


def test_all_zero_weight():
    W = np.zeros((128, 256), dtype=np.int8)
    A = bsp.UnionMatrix(_dev(W), 4)
    assert A.info()["total_values"] == 0
    Y = A.spmm(_dev(_acts(4, 256, 4, 1))).cpu().numpy()
    assert np.all(Y == 0)


def test_guard_bands():
    W = _weights(192, 256, 8, 0.5, 51)
    X = _acts(5, 256, 8, 52)
    A = bsp.UnionMatrix(_dev(W), 8)
    pad = 64
    buf = torch.full((pad + 5 * 192 + pad,), 12345, dtype=torch.int32, device=DEV)
    Y = buf[pad:pad + 5 * 192].view(5, 192)
    A.spmm(_dev(X), out=Y)
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 12345) and np.all(b[-pad:] == 12345)
    np.testing.assert_array_equal(Y.cpu().numpy().astype(np.int64), u.union_spmm(W, X))


def test_errors():
    L = bsp.lib()
    import ctypes
    h = ctypes.c_void_p()
    W = torch.zeros((64, 64), dtype=torch.int8, device=DEV)
    assert L.bsp_union_encode(W.data_ptr(), 5, 64, 64, None, ctypes.byref(h)) == 1    # bits
    assert L.bsp_union_encode(W.data_ptr(), 4, 64, 60, None, ctypes.byref(h)) == 2    # K % 16
    assert L.bsp_union_encode(W.data_ptr() + 1, 4, 64, 48, None, ctypes.byref(h)) == 4  # alignment
    Wk = torch.zeros((1, 1 << 21), dtype=torch.int8, device=DEV)
    assert L.bsp_union_encode(Wk.data_ptr(), 4, 1, 1 << 21, None, ctypes.byref(h)) == 2  # W4 K >= 2^21
    W8 = torch.full((64, 64), 9, dtype=torch.int8, device=DEV)
    assert L.bsp_union_encode(W8.data_ptr(), 4, 64, 64, None, ctypes.byref(h)) == 1   # outside int4
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits", [4, 8])
def test_llama7b_ffn_shape_sampled_rows(bits):
    """A 4096 x 11008 layer at 50%, N = 1, 8, 16; the oracle's product on
    four sampled rows of every 64-row strip."""
    M, K = 4096, 11008
    W = _weights(M, K, bits, 0.5, 300 + bits)
    X = _acts(16, K, bits, 301 + bits)
    rows = sample_rows(M, 4, seed=bits)
    ref = u.union_spmm(W[rows], X)
    A = bsp.UnionMatrix(_dev(W), bits)
    for N in (1, 8, 16):
        Y = A.spmm(_dev(X[:N])).cpu().numpy().astype(np.int64)
        np.testing.assert_array_equal(Y[:, rows], ref[:N])
    A.check()


def _paired_rows(M, K, bits, seed):
    """Weights whose rows come in identical-pattern pairs (2k, 2k + 1) with
    independent values: row reordering can halve the active union entries."""
    rng = np.random.default_rng(seed)
    lo, hi = -(1 << (bits - 1)), (1 << (bits - 1))
    pat = np.repeat(rng.random((M // 2, K)) < 0.3, 2, axis=0)
    vals = rng.integers(lo, hi - 1, size=(M, K))
    vals[vals >= 0] += 1
    return (vals * pat).astype(np.int8)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("kind", ["paired", "random"])
def test_reordered_encode_matches_oracle(bits, kind):
    W = _paired_rows(192, 320, bits, 61 + bits) if kind == "paired" else _weights(130, 208, bits, 0.6, 62 + bits)
    A = bsp.UnionMatrix(_dev(W), bits, reorder=True)
    assert A.info()["reordered"] == 1
    perms = A.perms().cpu().numpy().astype(np.int64)
    for p in perms:
        assert sorted(p.tolist()) == list(range(64))
    enc = u.union_encode(W, bits, perms=perms)
    masks, offsets, values = A.arrays()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(masks.cpu().numpy().view(np.uint64), enc["masks"])
    np.testing.assert_array_equal(offsets.cpu().numpy().view(np.uint32), enc["offsets"])
    np.testing.assert_array_equal(values.cpu().numpy(), u.pack_values(enc["values"], bits))
    assert A.storage_bytes() == u.storage_bytes(enc)
    np.testing.assert_array_equal(A.decode().cpu().numpy(), W)
    plain = u.union_encode(W, bits)
    assert int(enc["offsets"][-1]) <= int(plain["offsets"][-1])
    if kind == "paired":
        assert int(enc["offsets"][-1]) < int(plain["offsets"][-1])


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N", [1, 5, 16, 20])
def test_reordered_spmm_exact(bits, N):
    """Products of a reordered encoding come out in the original row order."""
    W = _paired_rows(256, 1024, bits, 70 + bits)
    X = _acts(N, 1024, bits, 71 + N)
    A = bsp.UnionMatrix(_dev(W), bits, reorder=True)
    Y = A.spmm(_dev(X)).cpu().numpy().astype(np.int64)
    A.check()
    np.testing.assert_array_equal(Y, u.union_spmm(W, X))


def test_reordered_split_k_forced(monkeypatch):
    W = _paired_rows(320, 1024, 8, 81)
    X = _acts(8, 1024, 8, 82)
    ref = u.union_spmm(W, X)
    A = bsp.UnionMatrix(_dev(W), 8, reorder=True)
    for sp in (1, 5, 16):
        tune("union_splitk", str(sp))
        np.testing.assert_array_equal(A.spmm(_dev(X)).cpu().numpy().astype(np.int64), ref)
    A.check()


def test_wait_that_runs_out_reports_timeout():
    """In the test build of the library (libbsp_test.so) each warp's producer
    skips its first tile's copies (a barrier nothing completes); the bounded
    wait gives up, the kernel records BSP_ERR_TIMEOUT, drains its other
    copies and returns; the next call is exact (workspace and counters were
    left clean)."""
    W = _weights(256, 1024, 8, 0.5, 91)
    X = _acts(4, 1024, 8, 92)
    with bsp.test_library() as T:
        A = bsp.UnionMatrix(_dev(W), 8)
        Xd = _dev(X)
        tune("union_splitk", 4)
        try:
            assert T.bsp_testing_set_stall(1) == 0 and T.bsp_testing_set_spin_cap(2000) == 0
            A.spmm(Xd)
            with pytest.raises(bsp.BspError) as e:
                A.check()
            assert e.value.status == 7
        finally:
            T.bsp_testing_set_stall(0)
            T.bsp_testing_set_spin_cap(0)
        A.check()  # cleared
        np.testing.assert_array_equal(A.spmm(Xd).cpu().numpy().astype(np.int64), u.union_spmm(W, X))
        A.check()
        A.close()
