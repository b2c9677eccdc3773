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
from helpers import assert_within_bound, to_dev_f16, tune

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


@pytest.mark.parametrize("splits", [1, 2, 5, 16])
def test_narrow_forced_splits(splits, monkeypatch):
    """16 GT columns: 16 splits is one column per CTA."""
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
