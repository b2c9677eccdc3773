"""GPU parity of the tcgen05 narrow kernel (fp16, N <= 16: one MMA of
N = 16 per K = 16, split-K through the handle's workspace) against the
oracle, on its own edge cases: one GT column, one split per GT column,
half and single-row tiles, and the dispatch threshold."""
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
def _narrow(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tune("narrow_min_n", "1")
    yield
    tune("narrow_min_n")
    tune("narrow_ctas")


def _run(W, X):
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    Y = A.spmm(to_dev_f16(X, DEV))
    A.check()
    return Y.cpu().numpy()


@pytest.mark.parametrize("M,K", [(128, 64),     # one tile, one GT column
                                 (64, 512),     # half tile (one GT row strip)
                                 (1, 8),        # one row, K padded to one GT column
                                 (200, 1000),   # ragged M and K
                                 (1024, 2048)])
@pytest.mark.parametrize("N", [1, 2, 7, 16])
def test_narrow_shapes(M, K, N):
    W = synth.weights_f16(M, K, 0.5, "uniform", 500 + M + K + N)
    X = synth.activations_f16(N, K, 501 + N)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(_run(W, X), Yref, S, f"narrow {M}x{K} N={N}")


@pytest.mark.parametrize("splits", [1, 2, 5, 16, 48])
def test_narrow_forced_splits(splits, monkeypatch):
    """3 tiles of 16 GT columns (48 steps) balanced over `splits` CTAs: 1 is
    one CTA taking the whole tiles one after another (both accumulators
    reused), 2, 5 and 16 split tiles between CTAs, 48 is one GT column per
    CTA."""
    M, K, N = 384, 1024, 12
    W = synth.weights_f16(M, K, 0.6, "uniform", 510)
    X = synth.activations_f16(N, K, 511)
    Yref, S = oracle.spmm_f16(W, X)
    tune("narrow_ctas", str(splits))
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    Xd = to_dev_f16(X, DEV)
    for _ in range(3):  # the workspace and counters are clean after each call
        assert_within_bound(A.spmm(Xd).cpu().numpy(), Yref, S, f"narrow splits={splits}")
    A.check()


@pytest.mark.parametrize("splits", [1, 3])
def test_narrow_runs_longer_than_offsets_window(splits):
    """64 GT columns on one or three CTAs: runs of 64 and about 22 steps of
    one tile, longer than the 32 offsets the producer's lane window holds,
    so the producer reloads the window inside a run."""
    M, K, N = 256, 4096, 5
    W = synth.weights_f16(M, K, 0.5, "uniform", 515 + splits)
    X = synth.activations_f16(N, K, 516)
    Yref, S = oracle.spmm_f16(W, X)
    tune("narrow_ctas", str(splits))
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    assert_within_bound(A.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, f"narrow long units {splits}")
    A.check()


def test_narrow_small_integers_exact(monkeypatch):
    tune("narrow_ctas", "3")
    W = synth.small_int_f16((256, 256), -8, 8, seed=521, sparsity=0.5)
    X = synth.small_int_f16((9, 256), -8, 8, seed=522)
    Yref, _ = oracle.spmm_f16(W, X)
    np.testing.assert_array_equal(_run(W, X).astype(np.float64), Yref)


def test_narrow_then_cores_share_workspace(monkeypatch):
    """Alternating the narrow and CUDA-core kernels on one handle: both
    leave the split-K workspace and counters zero for the other."""
    M, K = 512, 2048
    W = synth.weights_f16(M, K, 0.5, "uniform", 531)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    for i, N in enumerate((8, 16, 3, 16, 1, 8)):
        tune("narrow_min_n", "1" if i % 2 == 0 else "17")
        X = synth.activations_f16(N, K, 540 + i)
        Yref, S = oracle.spmm_f16(W, X)
        assert_within_bound(A.spmm(to_dev_f16(X, DEV)).cpu().numpy(), Yref, S, f"call {i} N={N}")
    A.check()


def test_narrow_guard_bands():
    W = synth.weights_f16(192, 256, 0.5, "uniform", 551)
    X = synth.activations_f16(3, 256, 552)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    pad = 64
    buf = torch.full((pad + 3 * 192 + pad,), 12345.0, dtype=torch.float16, device=DEV)
    Y = buf[pad:pad + 3 * 192].view(3, 192)
    A.spmm(to_dev_f16(X, DEV), out=Y)
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == np.float16(12345.0)) and np.all(b[-pad:] == np.float16(12345.0))
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y.cpu().numpy(), Yref, S, "narrow guard")


# ---- int8 weights on the tensor cores: exact fp16 copies of the int8 values
# and of X, fp32 runs of at most 16 GT columns (exact integers), int32 sums

def _run_i8(W, X):
    A = bsp.BitmapMatrix(to_dev(W, DEV))
    Y = A.spmm(to_dev(X, DEV))
    A.check()
    return Y.cpu().numpy().astype(np.int64)


@pytest.mark.parametrize("M,K", [(128, 64),     # one tile, one GT column
                                 (64, 512),     # half tile
                                 (1, 16),       # one row, K padded to one GT column
                                 (200, 1008),   # ragged M and K (16 GT columns: one run)
                                 (330, 1040),   # 17 GT columns: a run of 16 and one of 1
                                 (1024, 2048)])
@pytest.mark.parametrize("N", [1, 2, 7, 16])
def test_narrow_int8_exact(M, K, N):
    tune("narrow_min_n_i8", "1")
    W = synth.weights_i8(M, K, 0.5, 560 + M + K + N)
    X = synth.activations_i8(N, K, 561 + N)
    np.testing.assert_array_equal(_run_i8(W, X), oracle.spmm_i8(W, X))


def test_narrow_int8_extreme_values_exact():
    """Every weight 127 or -127 and every activation -128 or 127: a run of 16
    GT columns sums 1024 products of magnitude up to 16256, just below
    2^24, so the fp32 accumulator is exact only because runs stop at 16
    columns; 64 GT columns make four runs per tile."""
    M, K, N = 256, 4096, 16
    g = np.random.default_rng(570)
    W = np.where(g.random((M, K)) < 0.5, 127, -127).astype(np.int8)
    W[:, ::7] = 0
    X = np.where(g.random((N, K)) < 0.5, -128, 127).astype(np.int8)
    X[0, :] = -128  # column 0: |sums| at their largest
    W[0, :] = 127
    tune("narrow_min_n_i8", "1")
    np.testing.assert_array_equal(_run_i8(W, X), oracle.spmm_i8(W, X))


@pytest.mark.parametrize("splits", [1, 3, 16, 64])
def test_narrow_int8_forced_splits(splits):
    """3 tiles of 64 GT columns over 1 .. 64 CTAs: runs that start inside a
    CTA's first segment, segments shorter than a run, one column per CTA."""
    M, K, N = 384, 4096, 9
    W = synth.weights_i8(M, K, 0.6, 575)
    X = synth.activations_i8(N, K, 576)
    tune("narrow_min_n_i8", "1")
    tune("narrow_ctas", str(splits))
    A = bsp.BitmapMatrix(to_dev(W, DEV))
    Xd = to_dev(X, DEV)
    ref = oracle.spmm_i8(W, X)
    for _ in range(3):  # the int32 workspace is clean after each call
        np.testing.assert_array_equal(A.spmm(Xd).cpu().numpy().astype(np.int64), ref)
    A.check()


def test_narrow_int8_and_team_kernel_share_workspace():
    """Alternating the int8 narrow and team kernels on one handle."""
    M, K = 512, 2048
    W = synth.weights_i8(M, K, 0.5, 580)
    A = bsp.BitmapMatrix(to_dev(W, DEV))
    for i, N in enumerate((8, 16, 3, 16, 1, 8)):
        tune("narrow_min_n_i8", "1" if i % 2 == 0 else "17")
        X = synth.activations_i8(N, K, 590 + i)
        np.testing.assert_array_equal(A.spmm(to_dev(X, DEV)).cpu().numpy().astype(np.int64),
                                      oracle.spmm_i8(W, X))
    A.check()
