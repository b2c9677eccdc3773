"""Every product path can be captured into a CUDA graph and replayed: no
call allocates, synchronises or reads back inside bsp_spmm, bsp_spmspv or
bsp_union_spmm after a first call (which sets the kernels' shared-memory
attributes).  Each replay reads the current contents of X and must match
the oracle; the split-K workspace and counters stay consistent across
replays."""
import numpy as np
import pytest
import torch

import bitmap_encoded_unstructured_gb300 as bsp
import oracle
from oracle import ie_bme as u
from bitmap_encoded_unstructured_gb300 import synth
from helpers import assert_within_bound, to_dev_f16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _capture(fn):
    fn()  # first call outside the capture: per-device kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("N", [1, 2, 4, 5, 16, 40])
def test_spmm_graph_replay(N):
    """N = 1, 2: GT-per-warp kernel; 4: team kernel; 5, 16: narrow tcgen05
    kernel; 40: prefill tcgen05 kernel."""
    M, K = 512, 2048
    W = synth.weights_f16(M, K, 0.5, "uniform", 600 + N)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    Xd = torch.empty((N, K), dtype=torch.float16, device=DEV)
    Yd = torch.empty((N, M), dtype=torch.float16, device=DEV)
    X0 = synth.activations_f16(N, K, 601 + N)
    Xd.copy_(torch.from_numpy(X0.view(np.float16)))
    g = _capture(lambda: A.spmm(Xd, out=Yd))
    for r in range(3):
        X = synth.activations_f16(N, K, 610 + 10 * N + r)
        Xd.copy_(torch.from_numpy(X.view(np.float16)))
        g.replay()
        torch.cuda.synchronize()
        Yref, S = oracle.spmm_f16(W, X)
        assert_within_bound(Yd.cpu().numpy(), Yref, S, f"graph replay {r} N={N}")
    A.check()


def test_spmspv_graph_replay():
    M, K = 512, 4096
    W = synth.weights_f16(M, K, 0.5, "uniform", 620)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    xd = torch.empty(K, dtype=torch.float16, device=DEV)
    yd = torch.empty(M, dtype=torch.float16, device=DEV)
    xd.copy_(torch.from_numpy(synth.activations_relu_f16(K, 621).view(np.float16)))
    g = _capture(lambda: A.spmspv(xd, out=yd))
    for r in range(3):
        x = synth.activations_relu_f16(K, 630 + r)
        xd.copy_(torch.from_numpy(x.view(np.float16)))
        g.replay()
        torch.cuda.synchronize()
        yref, s = oracle.spmspv_f16(W, x)
        assert_within_bound(yd.cpu().numpy().reshape(1, -1), yref.reshape(1, -1), s.reshape(1, -1), f"spmspv {r}")
    A.check()


@pytest.mark.parametrize("bits", [4, 8])
def test_union_graph_replay(bits):
    M, K, N = 384, 2048, 8
    W = synth.weights_int(M, K, bits, 0.5, 640 + bits)
    A = bsp.UnionMatrix(torch.from_numpy(W).to(DEV), bits)
    Xd = torch.empty((N, K), dtype=torch.int8, device=DEV)
    Yd = torch.empty((N, M), dtype=torch.int32, device=DEV)
    Xd.copy_(torch.from_numpy(synth.activations_int(N, K, bits, 641)))
    g = _capture(lambda: A.spmm(Xd, out=Yd))
    for r in range(3):
        X = synth.activations_int(N, K, bits, 650 + r)
        Xd.copy_(torch.from_numpy(X))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(Yd.cpu().numpy().astype(np.int64), u.union_spmm(W, X))
    A.check()
