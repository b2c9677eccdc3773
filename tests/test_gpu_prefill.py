"""GPU parity of the tcgen05 prefill path (fp16, N > 16) against the oracle."""
import numpy as np
import pytest

import oracle
import bitmap_encoded_unstructured_gb300 as bsp
from bitmap_encoded_unstructured_gb300 import synth

from helpers import assert_within_bound, sample_rows, to_dev_f16, tune

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


DEV = torch.device("cuda:0")


def _run(W, X):
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    Y = A.spmm(to_dev_f16(X, DEV))
    A.check()
    return Y.cpu().numpy()


@pytest.mark.parametrize("M,K,N", [(128, 64, 32),      # one k-block, one ragged N tile
                                   (128, 320, 256),    # more k-blocks than stages
                                   (192, 256, 17),     # M % 128 == 64: half tile
                                   (384, 640, 300),    # two N tiles, the second ragged
                                   (256, 1024, 513),
                                   (512, 448, 300),    # four tiles, one ragged 512-column N tile
                                   (768, 640, 256),    # six tiles, one 256-column sub-tile
                                   (1024, 128, 40)])   # eight tiles, two k-blocks, narrow N
def test_prefill_small_shapes(M, K, N):
    W = synth.weights_f16(M, K, 0.5, "uniform", 300 + M + K + N)
    X = synth.activations_f16(N, K, 301 + N)
    Y = _run(W, X)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(Y, Yref, S, f"prefill {M}x{K} N={N}")


@pytest.mark.parametrize("M,K,N", [(128, 128, 32),     # KT = 2: one GT column per CTA of the cluster
                                   (192, 320, 17),     # KT = 5: 3 + 2; half tile
                                   (130, 136, 256),    # ragged M and K (KT = 3 over the padded grid)
                                   (768, 640, 256),
                                   (1024, 1024, 100)])
def test_prefill_split_k(M, K, N, monkeypatch):
    """Split-K over a cluster of two CTAs (rank 1's partial tile added in
    rank 0's shared memory) matches the oracle, forced on and forced off."""
    W = synth.weights_f16(M, K, 0.5, "uniform", 370 + M + K + N)
    X = synth.activations_f16(N, K, 371 + N)
    Yref, S = oracle.spmm_f16(W, X)
    tune("prefill_ksplit", "1")
    assert_within_bound(_run(W, X), Yref, S, f"split-K prefill {M}x{K} N={N}")
    tune("prefill_ksplit", "0")
    assert_within_bound(_run(W, X), Yref, S, f"prefill {M}x{K} N={N}")


@pytest.mark.parametrize("M,K,N", [(256, 512, 40), (1024, 2048, 256)])
def test_prefill_split_k_repeated(M, K, N, monkeypatch):
    """Twenty calls in a row (the cluster barriers of the exchange run
    every time): every result within the bound and all bitwise equal."""
    tune("prefill_ksplit", "1")
    W = synth.weights_f16(M, K, 0.5, "uniform", 390 + M)
    X = synth.activations_f16(N, K, 391)
    Yref, S = oracle.spmm_f16(W, X)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    Xd = to_dev_f16(X, DEV)
    outs = [A.spmm(Xd).clone() for _ in range(20)]
    A.check()
    for i, Y in enumerate(outs):
        assert torch.equal(Y, outs[0]), f"call {i} differs"
    assert_within_bound(outs[0].cpu().numpy(), Yref, S, f"split-K repeated {M}x{K} N={N}")


def test_prefill_split_k_small_integers_exact(monkeypatch):
    """Both partial sums and their sum are small integers: exact."""
    tune("prefill_ksplit", "1")
    W = synth.small_int_f16((256, 256), -8, 8, seed=381, sparsity=0.5)
    X = synth.small_int_f16((40, 256), -8, 8, seed=382)
    Yref, _ = oracle.spmm_f16(W, X)
    np.testing.assert_array_equal(_run(W, X).astype(np.float64), Yref)


def test_prefill_small_integers_exact():
    """Every partial sum is a small integer: one correct fp16 result."""
    W = synth.small_int_f16((256, 256), -8, 8, seed=311, sparsity=0.5)
    X = synth.small_int_f16((40, 256), -8, 8, seed=312)
    Y = _run(W, X).astype(np.float64)
    Yref, _ = oracle.spmm_f16(W, X)
    np.testing.assert_array_equal(Y, Yref)


@pytest.mark.parametrize("s", [0.0, 0.3, 0.7])
def test_prefill_sparsity_levels(s):
    W = synth.weights_f16(256, 512, s, "uniform" if s else "none", 320 + int(10 * s))
    X = synth.activations_f16(64, 512, 321)
    Yref, S = oracle.spmm_f16(W, X)
    assert_within_bound(_run(W, X), Yref, S, f"prefill s={s}")


def test_prefill_all_zero_weight():
    W = np.zeros((128, 256), dtype=np.uint16)
    X = synth.activations_f16(33, 256, 331)
    assert np.all(_run(W, X) == 0)
