"""GPU parity at the full sizes the benchmark times, on the benchmark's own
seeded inputs and launch configuration.

The oracle cannot compute whole full-size outputs in seconds, so it computes
sampled rows (every 64-row strip represented) and the GPU output is compared
on them: fp16 within |y - y_ref| <= 4e-3 * sum_k |w_mk x_kn| + 1e-5, int8 bit
for bit.  The shapes are the workloads of SpInfer's "Results" section and the
SPDP kernel evaluation (section 5.3): Llama-2-70B FFN prefill at N = 1024 and
4096 (two 256-column sub-tiles per CTA), the 8192 x 8192 sparsity sweep at 30%
and 70%, INT8 11008 x 4096 / 4096 x 11008 at 50% and 60%, and the IE-BME leg
(UnionSparse's W8A8 / W4A4 product, plain and row-reordered) on the OPT-13B
QKV and FC2 projections.
"""
import numpy as np
import pytest

import bench
import oracle
import bitmap_encoded_unstructured_gb300 as bsp

from helpers import assert_within_bound, sample_rows, to_dev, to_dev_f16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(autouse=True)
def _need_gpu():
    if DEV is None:
        pytest.skip("no CUDA device")


def _rows_of(Y, rows):
    """Y [N][M] on the device -> the sampled columns (rows of W) on the host."""
    idx = torch.from_numpy(rows).to(Y.device)
    return Y.index_select(1, idx).cpu().numpy()


@pytest.mark.parametrize("li", [0, 1])
def test_prefill_llama70b_ffn_full_size(li):
    """Llama-2-70B FFN up (28672 x 8192) and down (8192 x 28672) projections
    at 50%: N = 256 (one sub-tile, split-K pairs where chosen), 1024 and 4096
    (two sub-tiles per CTA), 2 sampled rows of every 64-row strip."""
    name, M, K = bench.PREFILL_LAYERS[li]
    W = bench.prefill_weights(name, M, K)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    rows = sample_rows(M, 2, seed=M + li)
    for N in bench.PREFILL_NS:
        X = bench.prefill_acts(N, K)
        Y = A.spmm(to_dev_f16(X, DEV))
        A.check()
        Yref, S = oracle.spmm_f16(W[rows], X)
        assert_within_bound(_rows_of(Y, rows), Yref, S, f"{name} N={N}")
        del Y
    A.close()


@pytest.mark.parametrize("s", [0.3, 0.7])
def test_sparsity_sweep_full_size(s):
    """The 8192 x 8192 sweep layer at its lowest and highest sparsity, every
    N the sweep times, 2 sampled rows per strip."""
    M, K = bench.SWEEP_SHAPE
    W = bench.sweep_weights(s)
    A = bsp.BitmapMatrix(to_dev_f16(W, DEV))
    rows = sample_rows(M, 2, seed=int(100 * s))
    for N in bench.SWEEP_NS:
        X = bench.sweep_acts(N)
        Y = A.spmm(to_dev_f16(X, DEV))
        A.check()
        Yref, Sref = oracle.spmm_f16(W[rows], X)
        assert_within_bound(_rows_of(Y, rows), Yref, Sref, f"sweep s={s} N={N}")
    A.close()


@pytest.mark.parametrize("s", bench.INT8_SPARSITY)
@pytest.mark.parametrize("li", [0, 1])
def test_int8_full_size(li, s):
    """INT8 bitmap SpMM at full size: the exact int32 product and the
    per-row dequantised fp32 product, bit for bit on 4 sampled rows of every
    strip, N = 1, 8, 16."""
    _, M, K = bench.INT8_LAYERS[li]
    W, X, scale = bench.int8_inputs(li, s)
    A = bsp.BitmapMatrix(to_dev(W, DEV))
    rows = sample_rows(M, 4, seed=7 * li + int(10 * s))
    acc = oracle.spmm_i8(W[rows], X)
    ref_scaled = oracle.scale_i8(acc, scale[rows])
    sd = to_dev(scale, DEV)
    for N in bench.INT8_NS:
        Xd = to_dev(X[:N].copy(), DEV)
        Y = A.spmm(Xd)
        Yf = A.spmm_scaled(Xd, sd)
        A.check()
        np.testing.assert_array_equal(_rows_of(Y, rows).astype(np.int64), acc[:N])
        np.testing.assert_array_equal(_rows_of(Yf, rows).view(np.uint32), ref_scaled[:N].view(np.uint32))
    A.close()


@pytest.mark.parametrize("bits,reorder", [(8, False), (4, False), (4, True)])
@pytest.mark.parametrize("li", [0, 3])
def test_ie_bme_full_size(li, bits, reorder):
    """The IE-BME leg's own configurations (UnionSparse): the OPT-13B QKV and
    FC2 projections as b-bit integers with i.i.d. 50% masks, W8A8, W4A4 and
    W4A4 with bitmap-aware row reordering, N = 1, 8, 16: the exact int32
    product, bit for bit on 2 sampled rows of every 64-row strip."""
    from bitmap_encoded_unstructured_gb300 import synth
    from oracle import ie_bme
    name, M, K = bench.LAYERS[li]
    W = synth.weights_int(M, K, bits, 0.5, synth.seed_for(6, 10 * bits + li), exact=False)
    A = bsp.UnionMatrix(to_dev(W, DEV), bits, reorder=reorder)
    rows = sample_rows(M, 2, seed=11 * li + bits)
    for N in bench.UNION_NS:
        X = synth.activations_int(N, K, bits, synth.seed_for(6, N))
        Y = A.spmm(to_dev(X, DEV))
        A.check()
        np.testing.assert_array_equal(_rows_of(Y, rows).astype(np.int64), ie_bme.union_spmm(W[rows], X),
                                      err_msg=f"{name} W{bits}A{bits} reorder={reorder} N={N}")
    A.close()
