"""Two host threads use the library at the same time, each on a fresh handle
and its own stream, from their first call on: the per-device one-time setup
(kernel attributes, tuning knobs read from the environment) is taken under a
lock, so concurrent first calls are safe, and distinct handles are
independent.  Every kernel family is covered (GT-per-warp, narrow tcgen05,
prefill, int8, IE-BME) with results checked against the oracle."""
import threading

import numpy as np
import pytest
import torch

import oracle
from oracle import ie_bme as u
import bitmap_encoded_unstructured_gb300 as bsp
from bitmap_encoded_unstructured_gb300 import synth

from helpers import within_bound

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(autouse=True)
def _need_gpu():
    if DEV is None:
        pytest.skip("no CUDA device")


def _worker(seed, results, i, barrier):
    try:
        torch.cuda.set_device(DEV)
        s = torch.cuda.Stream()
        M, K = 384, 1024
        W = synth.weights_f16(M, K, 0.5, "uniform", seed)
        W8 = synth.weights_i8(M, K, 0.5, seed + 1)
        Wi = synth.weights_int(M, K, 4, 0.5, seed + 2)
        Xs = {N: synth.activations_f16(N, K, seed + 10 + N) for N in (1, 2, 8, 16, 40)}
        X8 = synth.activations_i8(8, K, seed + 3)
        Xi = synth.activations_int(4, K, 4, seed + 4)
        ok = []
        barrier.wait()  # both threads make their first calls together
        with torch.cuda.stream(s):
            A = bsp.BitmapMatrix(torch.from_numpy(W.view(np.float16)).to(DEV), stream=s)
            B = bsp.BitmapMatrix(torch.from_numpy(W8).to(DEV), stream=s)
            U = bsp.UnionMatrix(torch.from_numpy(Wi).to(DEV), 4, stream=s)
            outs = {N: A.spmm(torch.from_numpy(X.view(np.float16)).to(DEV), stream=s) for N, X in Xs.items()}
            y8 = B.spmm(torch.from_numpy(X8).to(DEV), stream=s)
            yi = U.spmm(torch.from_numpy(Xi).to(DEV), stream=s)
        s.synchronize()
        for N, X in Xs.items():
            ref, S = oracle.spmm_f16(W, X)
            ok.append(bool(within_bound(outs[N].cpu().numpy(), ref, S).all()))
        ok.append(np.array_equal(y8.cpu().numpy().astype(np.int64), oracle.spmm_i8(W8, X8)))
        ok.append(np.array_equal(yi.cpu().numpy().astype(np.int64), u.union_spmm(Wi, Xi)))
        A.check(s)
        B.check(s)
        U.check(s)
        for h in (A, B, U):
            h.close()
        results[i] = all(ok)
    except Exception as e:  # reported by the test below
        results[i] = repr(e)


def _two_threads():
    results = [None, None]
    barrier = threading.Barrier(2)
    ts = [threading.Thread(target=_worker, args=(900 + 50 * i, results, i, barrier)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=300)
    return results


def test_two_threads_first_calls_at_once_fresh_process():
    """In a new process, so that both threads really make the library's first
    calls (kernel attribute setup, tuning knobs) at the same time."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_gpu_threads as t; r = t._two_threads(); print(r); sys.exit(0 if r == [True, True] else 1)"
            % (here, os.path.dirname(here)))
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout + p.stderr


def test_two_threads_in_this_process():
    assert _two_threads() == [True, True]
