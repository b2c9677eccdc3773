"""GPU parity of the Tiled-CBC column index (SPDP section 4.1) and of the
column-skipping spMspV that uses it (section 4.2), through the C ABI.

The index arrays must equal the oracle's byte for byte; products equal the
N = 1 product of W with the pruned activation vector: int8 exactly, fp16
within |y - y_ref| <= 4e-3 * sum_k |w_mk x_k| + 1e-5.
"""
import numpy as np
import pytest

import oracle
from oracle import tiled_cbc as cbc
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


def _mat(W):
    return bsp.BitmapMatrix(to_dev_f16(W, DEV) if W.dtype == np.uint16 else to_dev(W, DEV))


def _arrays_equal(A, W):
    off, ci, bm, vals = A.column_index_arrays()
    e = cbc.encode(W)
    np.testing.assert_array_equal(off.cpu().numpy().view(np.uint32), e["offsets"])
    np.testing.assert_array_equal(ci.cpu().numpy().view(np.uint32), e["colinfo"])
    np.testing.assert_array_equal(bm.cpu().numpy().view(np.uint64), e["bitmaps"])
    v = vals.cpu().numpy()
    np.testing.assert_array_equal(v.view(np.uint16) if W.dtype == np.uint16 else v, e["values"])
    assert A.column_index_bytes() == cbc.storage_bytes(e)


@pytest.mark.parametrize("M,K,s", [(256, 64, 0.5), (512, 256, 0.3), (300, 136, 0.7), (768, 1024, 0.5),
                                   (256, 128, 0.0), (256, 64, 1.0)])
def test_index_equals_oracle_fp16(M, K, s):
    W = synth.weights_f16(M, K, s, "uniform" if 0 < s < 1 else "none", 700 + M + K)
    if s == 1.0:
        W[:] = 0
    A = _mat(W)
    A.build_column_index()
    _arrays_equal(A, W)


@pytest.mark.parametrize("M,K,s", [(256, 128, 0.5), (1100, 400, 0.6)])
def test_index_equals_oracle_int8(M, K, s):
    W = synth.weights_i8(M, K, s, 710 + M)
    A = _mat(W)
    A.build_column_index()
    _arrays_equal(A, W)


def _relu(K, seed, shift=-1.0364):
    return synth.activations_relu_f16(K, seed, shift)


@pytest.mark.parametrize("M,K", [(256, 64), (512, 1024), (300, 136), (1024, 2048), (4096, 512)])
@pytest.mark.parametrize("kind", ["relu", "dense", "zero", "single"])
def test_spmspv_fp16(M, K, kind):
    W = synth.weights_f16(M, K, 0.5, "uniform", 720 + M + K)
    if kind == "relu":
        x = _relu(K, 721)
    elif kind == "dense":
        x = synth.activations_f16(1, K, 722)[0]
    elif kind == "zero":
        x = np.zeros(K, dtype=np.uint16)
    else:
        x = np.zeros(K, dtype=np.uint16)
        x[K // 3] = 0x3C00
    A = _mat(W)
    A.build_column_index()
    y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
    A.check()
    yref, S = oracle.spmm_f16(W, x.reshape(1, -1))
    assert_within_bound(y.reshape(1, -1), yref, S, f"cbc spmspv {kind} {M}x{K}")
    if kind == "zero":
        assert np.all(y.view(np.uint16) == 0)


@pytest.mark.parametrize("splits", [1, 2, 5, 64])
def test_spmspv_forced_splits(splits):
    """The split-K structure (one warp's run of GTile columns, partial sums
    in the workspace, the finishing kernel) at several split counts."""
    M, K = 768, 4096
    W = synth.weights_f16(M, K, 0.5, "uniform", 730)
    x = _relu(K, 731)
    A = _mat(W)
    A.build_column_index()
    yref, S = oracle.spmm_f16(W, x.reshape(1, -1))
    tune("splitk", splits)
    for _ in range(3):  # the workspace is left clean call after call
        y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
        assert_within_bound(y.reshape(1, -1), yref, S, f"cbc splits={splits}")
    A.check()


def test_spmspv_small_integers_exact():
    """Products and partial sums are small integers: one correct fp16."""
    M, K = 512, 256
    W = synth.small_int_f16((M, K), -8, 8, seed=740, sparsity=0.5)
    x = synth.small_int_f16((1, K), -8, 8, seed=741, sparsity=0.6)[0]
    A = _mat(W)
    A.build_column_index()
    tune("splitk", 3)
    y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy().view(np.uint16)
    yref, _ = oracle.spmm_f16(W, x.reshape(1, -1))
    np.testing.assert_array_equal(y, yref[0].astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("M,K", [(256, 128), (1100, 4096)])
def test_spmspv_int8_exact(M, K):
    W = synth.weights_i8(M, K, 0.5, 750 + M)
    x = synth.activations_i8(1, K, 751)[0]
    x[np.random.default_rng(752).random(K) < 0.8] = 0
    A = _mat(W)
    A.build_column_index()
    y = A.spmspv(to_dev(x, DEV)).cpu().numpy().astype(np.int64)
    A.check()
    np.testing.assert_array_equal(y, oracle.spmm_i8(W, x.reshape(1, -1))[0])


@pytest.mark.parametrize("tau", [0.0, 0.3, 1.0])
def test_spmspv_threshold(tau):
    """|x| <= tau pruned (NaN never): the product of W with the pruned x."""
    M, K = 512, 2048
    W = synth.weights_f16(M, K, 0.5, "uniform", 760)
    x = synth.activations_f16(1, K, 761)[0]
    A = _mat(W)
    A.build_column_index()
    y = A.spmspv_threshold(to_dev_f16(x, DEV), tau).cpu().numpy()
    xp = oracle.prune_activations_f16(x, tau)
    yref, S = oracle.spmm_f16(W, xp.reshape(1, -1))
    assert_within_bound(y.reshape(1, -1), yref, S, f"cbc threshold {tau}")


def test_spmspv_threshold_int8():
    M, K = 256, 1024
    W = synth.weights_i8(M, K, 0.5, 770)
    x = synth.activations_i8(1, K, 771)[0]
    A = _mat(W)
    A.build_column_index()
    y = A.spmspv_threshold(to_dev(x, DEV), 40.0).cpu().numpy().astype(np.int64)
    xp = oracle.prune_activations_i8(x, 40.0)
    np.testing.assert_array_equal(y, oracle.spmm_i8(W, xp.reshape(1, -1))[0])


def test_deterministic_mode_bit_identical():
    M, K = 1024, 8192
    W = synth.weights_f16(M, K, 0.5, "uniform", 780)
    x = _relu(K, 781)
    A = _mat(W)
    A.build_column_index()
    A.set_deterministic(True)
    xd = to_dev_f16(x, DEV)
    outs = [A.spmspv(xd).clone() for _ in range(8)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    yref, S = oracle.spmm_f16(W, x.reshape(1, -1))
    assert_within_bound(outs[0].cpu().numpy().reshape(1, -1), yref, S, "cbc deterministic")


def test_graph_capture_and_replay():
    """The column-skipping product allocates nothing once the index exists:
    it captures into a CUDA graph and replays correctly with new x."""
    M, K = 512, 2048
    W = synth.weights_f16(M, K, 0.5, "uniform", 790)
    A = _mat(W)
    A.build_column_index()
    xd = to_dev_f16(_relu(K, 791), DEV)
    y = torch.empty(M, dtype=torch.float16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A.spmspv(xd, out=y, stream=s)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        A.spmspv(xd, out=y, stream=s)
    for seed in (792, 793):
        x = _relu(K, seed)
        xd.copy_(to_dev_f16(x, DEV))
        g.replay()
        torch.cuda.synchronize()
        yref, S = oracle.spmm_f16(W, x.reshape(1, -1))
        assert_within_bound(y.cpu().numpy().reshape(1, -1), yref, S, f"graph replay {seed}")


def test_opt13b_fc2_full_size_sampled_rows():
    """The FC2 projection (5120 x 20480, 50% magnitude mask) with the
    post-ReLU activation of the benchmark (about 85% zeros): 4 sampled rows
    of every 64-row strip against the oracle."""
    M, K = 5120, 20480
    W = synth.weights_f16(M, K, 0.5, "magnitude", synth.seed_for(2, 3))
    x = synth.activations_relu_f16(K, synth.seed_for(2, 6))
    A = _mat(W)
    A.build_column_index()
    y = A.spmspv(to_dev_f16(x, DEV)).cpu().numpy()
    A.check()
    rows = sample_rows(M, 4, seed=3)
    yref, S = oracle.spmm_f16(W[rows], x.reshape(1, -1))
    assert_within_bound(y[rows].reshape(1, -1), yref, S, "fc2 cbc spmspv")
