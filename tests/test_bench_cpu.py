"""Host-side pieces of bench.py that need no GPU: the closed-form storage
the sparsity sweep reports equals the bytes of the oracle's encoding of the
same kind of weight (exact-count uniform masks), and the per-call
algorithmic bytes of the decode step count the encoded weight plus X and Y.
CPU only."""
import os
import sys

import numpy as np
import pytest

import oracle
from bitmap_encoded_unstructured_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("s", [0.0, 0.3, 0.5, 0.7, 1.0])
@pytest.mark.parametrize("M,K", [(64, 64), (128, 320), (256, 192)])
def test_sweep_closed_form_matches_the_oracle(M, K, s):
    W = synth.weights_f16(M, K, s, "uniform", 7 + M + K)
    enc = oracle.encode(W)
    nnz = int(np.count_nonzero(W))
    assert bench.sweep_closed_form(M, K, nnz) == oracle.storage_bytes(enc)
    # every kept N(0, 0.02) draw is a nonzero fp16 at these sizes, so the
    # nominal count gives the same bytes
    assert nnz == M * K - round(s * M * K)
    assert bench.sweep_nominal_bytes(M, K, s) == oracle.storage_bytes(enc)


def test_sweep_closed_form_counts_the_stored_values():
    """Where some draws round to an fp16 zero (not stored), the closed form
    from the measured count still equals the oracle's bytes exactly, and the
    nominal estimate is above it by 2 bytes per such zero."""
    M, K, s = 512, 512, 0.5
    W = synth.weights_f16(M, K, s, "uniform", 11)
    W[np.nonzero(W)[0][:5], np.nonzero(W)[1][:5]] = 0  # five kept values become zeros
    nnz = int(np.count_nonzero(W))
    enc = oracle.encode(W)
    assert bench.sweep_closed_form(M, K, nnz) == oracle.storage_bytes(enc)
    assert bench.sweep_nominal_bytes(M, K, s) - oracle.storage_bytes(enc) == 2 * 5


def test_decode_step_bytes_count_weight_x_and_y():
    Ws = {"out": synth.weights_f16(5120, 5120, 0.5, "uniform", 3)}
    relu = synth.activations_relu_f16(20480, 4)
    bpc, stor, _ = bench.algorithmic_bytes(Ws, relu)
    enc_bytes = oracle.storage_bytes(oracle.encode(Ws["out"]))
    assert stor["out"] == enc_bytes
    for N in bench.NS:
        assert bpc[("out", N)] == enc_bytes + 2 * 5120 * N + 2 * 5120 * N


def test_step_kernel_follows_the_dispatch(monkeypatch):
    monkeypatch.delenv("BSP_NARROW_MIN_N", raising=False)
    got = {N: bench.step_kernel(("qkv", N)) for N in (1, 2, 3, 4, 5, 8, 16)}
    assert got == {1: "spmm_decode_gtw_kernel", 2: "spmm_decode_gtw_kernel", 3: "spmm_narrow_kernel",
                   4: "spmm_narrow_kernel", 5: "spmm_narrow_kernel", 8: "spmm_narrow_kernel",
                   16: "spmm_narrow_kernel"}
    assert bench.step_kernel(("fc2", "spmspv")) == "spmspv_cbc_kernel"
    monkeypatch.setenv("BSP_NARROW_MIN_N", "17")
    assert bench.step_kernel(("qkv", 16)) == "spmm_decode_kernel"


def test_step_kernel_default_is_the_librarys():
    """bench.step_kernel labels the step's launches with the library's
    default fp16 dispatch threshold, read here from its source."""
    import re
    src = open(os.path.join(ROOT, "bitmap_encoded_unstructured_gb300", "csrc", "bsp_tuning.cu")).read()
    m = re.search(r"#define\s+BSP_NARROW_MIN_N_DEFAULT\s+(\d+)", src)
    assert m and int(m.group(1)) == bench.NARROW_MIN_N_DEFAULT


def test_spmspv_bytes_follow_the_oracle_fetch_accounting():
    """The bench's algorithmic bytes of the column-skipping spMspV are the
    oracle's fetched index bytes (ColInfo of every GTile, bitmaps and values
    of the active columns; here every GTile has an active column) plus the
    TileOffset, x and y."""
    from oracle import tiled_cbc
    M, K = 512, 1024
    W = synth.weights_f16(M, K, 0.5, "uniform", 21)
    x = synth.activations_relu_f16(K, 22)
    e = tiled_cbc.encode(W)
    act = (x & 0x7FFF) != 0
    expect = 4 * (e["NGT"] + 1) + tiled_cbc.fetched_bytes(e, act) + 2 * K + 2 * M
    assert bench.cbc_spmspv_bytes(W, x) == expect


def test_step_launch_count_includes_the_finishing_kernels():
    """gpu_launches counts a finishing kernel after every narrow and
    column-index spMspV call: on a 152-SM GB300 (304 narrow CTAs) every
    layer of the step has a tile whose steps are shared by two CTAs of the
    balanced partition, and FC2's 320 GTile columns make 160 spMspV splits."""
    P = 2 * 152
    for _, M, K in bench.LAYERS:
        KT, tiles = K // 64, -(-M // 128)
        T = tiles * KT
        owner = lambda x: ((x + 1) * min(P, T) - 1) // T  # noqa: E731  (the partition's owner of step x)
        assert any(owner(t * KT) != owner((t + 1) * KT - 1) for t in range(tiles))
    fc2_cols = dict((l[0], l) for l in bench.LAYERS)["fc2"][2] // 64
    assert -(-fc2_cols // 2) > 1
    per_step = sum(bench.LAUNCHES_PER_CALL[bench.step_kernel((name, N))]
                   for N in bench.NS for name, _, _ in bench.LAYERS) + bench.LAUNCHES_PER_CALL["spmspv_cbc_kernel"]
    assert per_step == 8 * 1 + 8 * 2 + 2


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the oracle on the host's cores, no GPU)
    prints one JSON line with the keys the driver reads, the reference-arm
    additions included (impl, cpu_baseline with kind/cores/sample and the
    line's value, e2e with zero transfer bytes)."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["metric"] == bench.METRIC and d["config"]["workload"] == bench._config()["workload"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["sample"] and c["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
