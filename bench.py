"""Benchmark: bitmap-SpMM decode GB/s (fraction of HBM peak) at N = 1..16.

Workload: the four projections of an OPT-13B decoder layer (QKV 15360x5120,
out 5120x5120, FC1 20480x5120, FC2 5120x20480), fp16, 50% magnitude-style
unstructured mask, synthetic N(0, 0.02) weights (no checkpoints needed).
One step = bsp_spmm on every layer at N = 1, 2, 8, 16, plus bsp_spmspv on
FC2 with a post-ReLU activation (~85% zeros) over FC2's Tiled-CBC column
index: 17 calls of the decode kernels.  The step's working set (354 MB of encoded weights) is larger than
L2 (129 MB), and each layer is re-read only after the three others have
passed through L2.

GB/s counts algorithmic bytes: the encoded weight (Stor) + X + Y for each
spmm; for the spMspV the column index's TileOffset and ColInfo rows, the
bitmaps and values of the active columns, x and y.

``--impl reference`` times the CPU oracle instead, on a bounded row sample
of the same workload, and prints the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bitmap_encoded_unstructured_gb300 import synth  # noqa: E402

LAYERS = [("qkv", 15360, 5120), ("out", 5120, 5120), ("fc1", 20480, 5120), ("fc2", 5120, 20480)]
NS = (1, 2, 8, 16)
# Llama-2-70B FFN projections for the prefill leg (fp16, 50% uniform mask)
PREFILL_LAYERS = [("llama_up", 28672, 8192), ("llama_down", 8192, 28672)]
PREFILL_NS = (256, 1024, 4096)
METRIC = "bitmap-SpMM decode GB/s (% of HBM peak) at N=1-16; prefill TFLOP/s"
# INT8 bitmap SpMM: W 11008x4096 and 4096x11008, nonzeros uniform in
# [-127, 127] \ {0}, 50% and 60% uniform masks, int8 X, N = 1, 8, 16
INT8_LAYERS = [("int8_11008x4096", 11008, 4096), ("int8_4096x11008", 4096, 11008)]
INT8_SPARSITY = (0.5, 0.6)
INT8_NS = (1, 8, 16)
# kernels of the decode step and their sources (with the dispatch): fp16
# N <= 2 on the GT-per-warp kernel, N >= 3 on the narrow tcgen05 kernel, the
# spMspV on the column-skipping kernel over the Tiled-CBC index (a narrow or
# spMspV call's finishing kernel, which converts split partial sums, is part
# of the same call)
STEP_KERNELS = "spmm_decode_gtw_kernel (N<=2) + spmm_narrow_kernel (N=8, 16) + spmspv_cbc_kernel (spMspV)"
STEP_SOURCES = ("spmm_decode.cu", "spmm_narrow.cu", "tiled_cbc.cu", "bsp_api.cu", "bsp_tuning.cu")
NARROW_MIN_N_DEFAULT = 3  # BSP_NARROW_MIN_N_DEFAULT of bsp_tuning.cu (a CPU test holds them equal)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0


# Kernels one call of the step launches: the narrow and column-index spMspV
# products are followed by their finishing kernel whenever tiles are split
# between CTAs, which holds for every layer of the step at the automatic
# CTA / split counts (tests/test_bench_cpu.py checks the split counts).
LAUNCHES_PER_CALL = {"spmm_decode_gtw_kernel": 1, "spmm_decode_kernel": 1, "spmm_narrow_kernel": 2,
                     "spmspv_cbc_kernel": 2}


def step_kernel(key):
    """The kernel a call of the step launches, by the library's fp16
    dispatch (BSP_NARROW_MIN_N, else the library's default)."""
    _, N = key
    if N == "spmspv":
        return "spmspv_cbc_kernel"
    if N <= 2:
        return "spmm_decode_gtw_kernel"
    min_n = int(os.environ.get("BSP_NARROW_MIN_N", str(NARROW_MIN_N_DEFAULT)))
    return "spmm_narrow_kernel" if N >= min_n else "spmm_decode_kernel"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _tensor_peak():
    """Dense fp16 tensor peak: the measured bf16 burst figure (fp16 and bf16
    have the same nominal dense rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (bf16 burst, same nominal rate as fp16)"
    return FALLBACK_TFLOPS, "fallback"


def prefill_weights(name, M, K):
    i = [l[0] for l in PREFILL_LAYERS].index(name)
    return synth.weights_f16(M, K, 0.5, "uniform", synth.seed_for(4, i))


def prefill_acts(N, K):
    return synth.activations_f16(N, K, synth.seed_for(4, 2))


def int8_inputs(li, s):
    """Seeded inputs of one INT8 configuration: layer index li of
    INT8_LAYERS, sparsity s: (W int8 [M][K], X int8 [16][K], row scales
    fp32 [M])."""
    _, M, K = INT8_LAYERS[li]
    W = synth.weights_i8(M, K, s, synth.seed_for(5, 2 * li + INT8_SPARSITY.index(s)))
    X = synth.activations_i8(max(INT8_NS), K, synth.seed_for(5, 4 + li))
    return W, X, synth.row_scales(M, synth.seed_for(5, 6 + li))


def sweep_weights(s):
    """Seeded weight of one sparsity-sweep point: fp16 bits [8192][8192] at
    sparsity s (uniform exact-count mask)."""
    M, K = SWEEP_SHAPE
    return synth.weights_f16(M, K, s, "uniform", synth.seed_for(2, round(s * 10)))


def sweep_acts(N):
    """Seeded activations of the sparsity sweep: fp16 bits [N][8192]."""
    return synth.activations_f16(N, SWEEP_SHAPE[1], synth.seed_for(2, N))


def make_workload(only=None):
    """Host-side synthetic inputs (numpy, seeded)."""
    Ws, xs = {}, {}
    for i, (name, M, K) in enumerate(LAYERS):
        if only and name not in only:
            continue
        Ws[name] = synth.weights_f16(M, K, 0.5, "magnitude", synth.seed_for(2, i))
        xs[name] = synth.activations_f16(16, K, synth.seed_for(2, 10 + i))
    relu = synth.activations_relu_f16(LAYERS[3][2], synth.seed_for(2, 6))
    return Ws, xs, relu


def cbc_spmspv_bytes(W, x):
    """Algorithmic bytes of the column-skipping spMspV over the Tiled-CBC
    index (256 x 64 GTiles): the TileOffset and the whole ColInfo row of
    every GTile with an active column, the four bitmap words (32 B) and the
    values of every active column tile, x and y."""
    M, K = W.shape
    tr, tc = -(-M // 256), -(-K // 64)
    act = np.zeros(tc * 64, dtype=bool)
    act[:K] = (x.view(np.uint16) & 0x7FFF) != 0
    nz = np.zeros((tr * 256, tc * 64), dtype=bool)
    nz[:M, :K] = W.view(np.uint16) != 0
    col_nnz = nz.reshape(tr, 256, tc * 64).sum(axis=1)           # [tr][columns]
    act_tiles = act.reshape(tc, 64).any(axis=1)                  # GTile columns with an active column
    n_gt = tr * int(act_tiles.sum())
    vals = int(col_nnz[:, act].sum())
    return 4 * (n_gt + 1) + 4 * 64 * n_gt + 32 * tr * int(act.sum()) + 2 * vals + 2 * K + 2 * M


def algorithmic_bytes(Ws, relu):
    """Per-call algorithmic bytes for each (layer, N) and for the spMspV."""
    out = {}
    stor = {}
    for name, M, K in LAYERS:
        if name not in Ws:
            continue
        nnz = int(np.count_nonzero(Ws[name]))
        ngt, nbt = (M // 64) * (K // 64), M * K // 64
        stor[name] = 4 * (ngt + 1) + 8 * nbt + 2 * nnz
        for N in NS:
            out[(name, N)] = stor[name] + 2 * K * N + 2 * M * N
    name, M, K = LAYERS[3]
    if name not in Ws:
        return out, stor, 0.0
    W = Ws[name]
    # the spMspV runs over the FC2 handle's Tiled-CBC column index
    out[("fc2", "spmspv")] = cbc_spmspv_bytes(W, relu)
    act = (relu.view(np.uint16) & 0x7FFF) != 0
    return out, stor, float(act.mean())


class ClockSampler:
    """nvidia-smi samples during the timed region (clocks, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.split(", ") for l in self.lines if l and not l.startswith("index")]
        rows = [r for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "samples": len(rows), "reasons": reasons}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _progress(msg: str) -> None:
    """One progress line on stderr (the JSON result goes to stdout)."""
    print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def _max_over_ranks(v: float, ws: int) -> float:
    """Max of a per-rank value over all ranks (the whole-job time)."""
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- CPU oracle timing

def _oracle_pass(Ws, xs, relu, bytes_per_call, rows_per_layer):
    """One pass of the step on the oracle over the first rows of each layer;
    (seconds, equivalent algorithmic bytes: each call's bytes times its row
    fraction)."""
    import oracle
    t0 = time.perf_counter()
    eq_bytes = 0.0
    for N in NS:
        for name, M, K in LAYERS:
            r = min(rows_per_layer, M)
            oracle.spmm_f16(Ws[name][:r], xs[name][:N])
            eq_bytes += bytes_per_call[(name, N)] * r / M
    name, M, K = LAYERS[3]
    r = min(rows_per_layer, M)
    oracle.spmm_f16(Ws[name][:r], relu.reshape(1, -1))
    eq_bytes += bytes_per_call[("fc2", "spmspv")] * r / M
    return time.perf_counter() - t0, eq_bytes


def time_oracle(Ws, xs, relu, bytes_per_call, stor, rows_per_layer=128, target_s=None):
    """The oracle on a bounded row sample of the whole step; GB/s of the
    equivalent algorithmic bytes.  With target_s, a first pass of
    rows_per_layer rows sizes a second, timed pass to about target_s
    seconds (rows capped at each layer's M)."""
    import oracle
    oracle.build()
    dt, eq = _oracle_pass(Ws, xs, relu, bytes_per_call, rows_per_layer)
    rows, passes = rows_per_layer, 1
    if target_s:
        rows = max(rows_per_layer, int(rows_per_layer * target_s / max(dt, 1e-6)))
        dt, eq = _oracle_pass(Ws, xs, relu, bytes_per_call, rows)
        while dt < 0.8 * target_s:  # rows capped at M: repeat the pass
            d2, e2 = _oracle_pass(Ws, xs, relu, bytes_per_call, rows)
            dt, eq, passes = dt + d2, eq + e2, passes + 1
    return {"value": eq / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 3), "rows_per_layer": rows, "passes": passes,
            "sample": f"first min({rows}, M) rows of each layer, every N in {list(NS)} plus the FC2 "
                      f"spMspV, {passes} pass(es) of the step on that row fraction; fp64 dense triple "
                      f"loop over fp16 inputs"}


def time_oracle_extra(Ws, xs, relu, bytes_per_call, stor, target_s=5.0):
    """Beside the all-cores figure: the same oracle product pinned to one
    thread on a row sample sized to about target_s seconds, and the
    oracle's encoder on the out-projection (5120 x 5120), whole."""
    import oracle
    oracle.build()
    n_all = oracle.num_threads()
    oracle.set_threads(1)
    try:
        one = time_oracle(Ws, xs, relu, bytes_per_call, stor, rows_per_layer=8, target_s=target_s)
    finally:
        oracle.set_threads(n_all)
    W = Ws["out"]
    t0 = time.perf_counter()
    enc = oracle.encode(W)
    enc_s = time.perf_counter() - t0
    return {"single_thread_value": one["value"], "single_thread_cores": 1,
            "single_thread_seconds": one["seconds"], "single_thread_rows_per_layer": one["rows_per_layer"],
            "encode_seconds": round(enc_s, 3), "encode_layer": "out 5120x5120 fp16 50% magnitude",
            "encode_MB_per_s": round(W.nbytes / enc_s / 1e6, 2),
            "encode_storage_bytes": int(oracle.storage_bytes(enc))}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    Ws, xs, relu = make_workload()
    bpc, stor, _ = algorithmic_bytes(Ws, relu)
    vals = []
    for i in range(args.warmup + args.steps):
        r = time_oracle(Ws, xs, relu, bpc, stor, rows_per_layer=16)
        if i >= args.warmup:
            vals.append(r)
    value = statistics.median(v["value"] for v in vals)
    secs = sum(v["seconds"] for v in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / len(vals) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _config(),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"]},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def _config():
    return {"workload": "OPT-13B decoder projections (QKV 15360x5120, out 5120x5120, FC1 20480x5120, "
                        "FC2 5120x20480), fp16, 50% magnitude mask; bsp_spmm at N=1,2,8,16 + FC2 "
                        "bsp_spmspv with ~85%-zero post-ReLU x",
            "sparsity": 0.5, "batch_n": list(NS), "group_tile": [64, 64],
            "l2": "inputs larger than L2: 354 MB of encoded weights rotate through a 129 MB L2 each step",
            "timing": "value: K steps with no events between calls; roofline and breakdown: a second K-step "
                      "pass with a CUDA event after every call",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- GPU arm

def run_case(args):
    """One (layer, N) configuration only, for profiler captures: encode the
    layer, run `warmup + steps` calls of bsp_spmm (or bsp_spmspv with N=0)."""
    import torch
    import bitmap_encoded_unstructured_gb300 as bsp
    layer, n = args.case.split(":")
    N = int(n)
    dev = torch.device("cuda", 0)
    if layer[:3] in ("w4_", "w8_"):  # IE-BME: w4_qkv:8 = W4A4 on the QKV projection, N = 8
        bits, lname = int(layer[1]), layer[3:]
        (name, M, K), = [l for l in LAYERS if l[0] == lname]
        A = bsp.UnionMatrix(torch.from_numpy(synth.weights_int(M, K, bits, 0.5, synth.seed_for(6, bits),
                                                               exact=False)).to(dev), bits)
        X = torch.from_numpy(synth.activations_int(N, K, bits, synth.seed_for(6, N))).to(dev)
        Y = torch.empty((N, M), dtype=torch.int32, device=dev)
        for _ in range(args.warmup):
            A.spmm(X, out=Y)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            A.spmm(X, out=Y)
        e.record()
        torch.cuda.synchronize()
        A.check()
        us = s.elapsed_time(e) * 1e3 / args.steps
        b = A.storage_bytes() + K * N + 4 * M * N
        print(json.dumps({"case": args.case, "us_per_call": round(us, 2), "GBps": round(b / us / 1e3, 1),
                          "note": "same layer every call"}))
        return 0
    if layer in dict((l[0], l) for l in PREFILL_LAYERS):
        (name, M, K), = [l for l in PREFILL_LAYERS if l[0] == layer]
        A = bsp.BitmapMatrix(torch.from_numpy(prefill_weights(name, M, K).view(np.float16)).to(dev))
        X = torch.from_numpy(synth.activations_f16(N, K, synth.seed_for(4, 2)).view(np.float16)).to(dev)
        Y = torch.empty((N, M), dtype=torch.float16, device=dev)
        for _ in range(args.warmup):
            A.spmm(X, out=Y)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            A.spmm(X, out=Y)
        e.record()
        torch.cuda.synchronize()
        A.check()
        us = s.elapsed_time(e) * 1e3 / args.steps
        tf = 2.0 * M * K * N / (us * 1e-6) / 1e12
        print(json.dumps({"case": args.case, "us_per_call": round(us, 2), "TFLOPs": round(tf, 1),
                          "frac_tensor_peak": round(tf / _tensor_peak()[0], 4)}))
        return 0
    if layer in dict((l[0], l) for l in INT8_LAYERS):  # int8_11008x4096:8 = the C5 layer at 50%, N = 8
        li = [l[0] for l in INT8_LAYERS].index(layer)
        _, M, K = INT8_LAYERS[li]
        W, X8, _ = int8_inputs(li, INT8_SPARSITY[0])
        A = bsp.BitmapMatrix(torch.from_numpy(W).to(dev))
        X = torch.from_numpy(X8[:N].copy()).to(dev)
        Y = torch.empty((N, M), dtype=torch.int32, device=dev)
        for _ in range(args.warmup):
            A.spmm(X, out=Y)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(args.steps):
            A.spmm(X, out=Y)
        e.record()
        torch.cuda.synchronize()
        A.check()
        us = s.elapsed_time(e) * 1e3 / args.steps
        b = A.storage_bytes() + K * N + 4 * M * N
        print(json.dumps({"case": args.case, "us_per_call": round(us, 2), "GBps": round(b / us / 1e3, 1),
                          "note": "same layer every call: L2-warm for layers under 129 MB"}))
        return 0
    Ws, xs, relu = make_workload(only={layer})
    (name, M, K), = [l for l in LAYERS if l[0] == layer]
    A = bsp.BitmapMatrix(torch.from_numpy(Ws[name].view(np.float16)).to(dev))
    if N == 0:
        x = torch.from_numpy(relu.view(np.float16)).to(dev) if name == "fc2" else \
            torch.from_numpy(xs[name][0].view(np.float16).copy()).to(dev)
        A.build_column_index()
        y = torch.empty(M, dtype=torch.float16, device=dev)
        fn = lambda: A.spmspv(x, out=y)
    else:
        X = torch.from_numpy(xs[name][:N].view(np.float16).copy()).to(dev)
        Y = torch.empty((N, M), dtype=torch.float16, device=dev)
        fn = lambda: A.spmm(X, out=Y)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        fn()
    e.record()
    torch.cuda.synchronize()
    A.check()
    us = s.elapsed_time(e) * 1e3 / args.steps
    stor = A.storage_bytes()
    b = stor + 2 * K * max(N, 1) + 2 * M * max(N, 1)
    print(json.dumps({"case": args.case, "us_per_call": round(us, 2), "GBps": round(b / us / 1e3, 1),
                      "note": "same layer every call: L2-warm for layers under 129 MB"}))
    return 0


def run_gpu(args):
    import torch
    import bitmap_encoded_unstructured_gb300 as bsp

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    Ws, xs, relu = make_workload()
    bpc, stor, act_frac = algorithmic_bytes(Ws, relu)
    mats = {}
    Xd, Yd = {}, {}
    for name, M, K in LAYERS:
        mats[name] = bsp.BitmapMatrix(torch.from_numpy(Ws[name].view(np.float16)).to(dev))
        assert mats[name].storage_bytes() == stor[name]
        Xd[name] = torch.from_numpy(xs[name].view(np.float16)).to(dev)
        Yd[name] = torch.empty((16, M), dtype=torch.float16, device=dev)
    mats["fc2"].build_column_index()  # the step's spMspV skips inactive columns
    xr = torch.from_numpy(relu.view(np.float16)).to(dev)
    yr = torch.empty(LAYERS[3][1], dtype=torch.float16, device=dev)
    Xn = {(name, N): Xd[name][:N].contiguous() for name, _, _ in LAYERS for N in NS}
    Yn = {(name, N): torch.empty((N, M), dtype=torch.float16, device=dev) for name, M, _ in LAYERS for N in NS}

    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    calls = []
    for N in NS:
        for name, _, _ in LAYERS:
            calls.append(((name, N), lambda name=name, N=N: bsp.bsp_spmm(
                mats[name].h, Xn[(name, N)].data_ptr(), N, Yn[(name, N)].data_ptr(), sh)))
    calls.append((("fc2", "spmspv"), lambda: bsp.bsp_spmspv(mats["fc2"].h, xr.data_ptr(), yr.data_ptr(), sh)))

    def step(events=None):
        for i, (_, fn) in enumerate(calls):
            fn()
            if events is not None:
                events[i].record(stream)

    _progress("decode step")
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    n_calls = len(calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_calls)] for _ in range(args.steps)]
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    _barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # the timed region of `value`: K steps with no instrumentation between
    # the calls (an event recorded between two launches ends the overlap of
    # programmatic dependent launch: measured 645 against 583 us per step)
    start.record(stream)
    for s in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    _barrier(ws)
    total_ms = start.elapsed_time(end)
    total_ms = _max_over_ranks(total_ms, ws)
    # a second timed pass of K steps with an event after every call: the
    # per-launch durations of the roofline (each call then runs without
    # overlap with the next, so these durations are the conservative ones)
    torch.cuda.synchronize()
    for s in range(args.steps):
        ev0[s].record(stream)
        step(ev[s])
    torch.cuda.synchronize()
    _barrier(ws)
    clk = clocks.stop()

    # per-launch durations from consecutive events on the launching stream
    per_call = {k: [] for k, _ in calls}
    for s in range(args.steps):
        prev = ev0[s]
        for i, (k, _) in enumerate(calls):
            per_call[k].append(prev.elapsed_time(ev[s][i]))
            prev = ev[s][i]
    step_bytes = sum(bpc[k] for k, _ in calls)
    value = ws * step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    launch_ms = sum(statistics.mean(v) for v in per_call.values())
    achieved = step_bytes / (launch_ms * 1e-3) / 1e9
    # per kernel: algorithmic bytes and mean launch time of its calls; the
    # dominant kernel (largest share of the launch time) gives the roofline
    by_kernel = {}
    for k, _ in calls:
        e = by_kernel.setdefault(step_kernel(k), {"launches": 0, "bytes": 0, "ms": 0.0})
        e["launches"] += 1
        e["bytes"] += bpc[k]
        e["ms"] += statistics.mean(per_call[k])
    dom = max(by_kernel, key=lambda n: by_kernel[n]["ms"])

    breakdown = {}
    for N in NS:
        b = sum(bpc[(n, N)] for n, _, _ in LAYERS)
        t = sum(statistics.median(per_call[(n, N)]) for n, _, _ in LAYERS)
        breakdown[f"N={N}"] = {
            "GBps": round(b / (t * 1e-3) / 1e9, 1), "frac_hbm": round(b / (t * 1e-3) / 1e9 / peak, 4),
            "us_per_layer": {n: round(statistics.median(per_call[(n, N)]) * 1e3, 2) for n, _, _ in LAYERS}}
    t_sp = statistics.median(per_call[("fc2", "spmspv")])
    breakdown["spmspv_fc2"] = {"GBps": round(bpc[("fc2", "spmspv")] / (t_sp * 1e-3) / 1e9, 1),
                               "us": round(t_sp * 1e3, 2), "active_columns": round(act_frac, 4),
                               "column_index_bytes": mats["fc2"].column_index_bytes(),
                               "speedup_vs_spmm_n1": round(statistics.median(per_call[("fc2", 1)]) / t_sp, 3)}

    traffic = None
    traffic_kernels = {}
    tp = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(tp):
        with open(tp) as f:
            tr = json.load(f)
        if tr.get("kernel_source_hash") == _kernel_hash():
            traffic_kernels = tr.get("kernels", {})
            traffic = traffic_kernels.get(dom, {}).get("dram_bytes_per_launch")

    # ---- e2e: same step through the host-buffer C-ABI call
    e2e = None
    if not args.no_e2e:
        _progress("e2e")
        Xh = {(n, N): torch.from_numpy(xs[n][:N].view(np.float16).copy()).pin_memory() for n, _, _ in LAYERS for N in NS}
        Yh = {(n, N): torch.empty((N, M), dtype=torch.float16).pin_memory() for n, M, _ in LAYERS for N in NS}
        h2d = sum(Xh[k].numel() * 2 for k in Xh)
        d2h = sum(Yh[k].numel() * 2 for k in Yh)
        # two streams, each layer's handle on one of them (a handle's calls stay
        # on one stream: its staging buffers are reused in stream order), so
        # one layer's copies overlap another layer's product
        e2e_streams = [stream, torch.cuda.Stream(dev)]
        lstream = {n: e2e_streams[i % 2] for i, (n, _, _) in enumerate(LAYERS)}

        def e2e_step():
            # the public host-buffer call, enqueued per layer and N; the step
            # ends when its results are in host memory
            for (n, N) in Xh:
                mats[n].spmm_host_async(Xh[(n, N)], Yh[(n, N)], stream=lstream[n].cuda_stream)
            for st in e2e_streams:
                st.synchronize()
        for _ in range(3):
            e2e_step()
        _barrier(ws)
        t0 = time.perf_counter()
        reps = max(3, args.steps // 5)
        for _ in range(reps):
            e2e_step()
        dt = _max_over_ranks(time.perf_counter() - t0, ws)
        e2e_bytes = sum(bpc[k] for k in Xh)
        # the blocking call (a stream synchronisation after every call), as before
        t1 = time.perf_counter()
        for _ in range(reps):
            for (n, N) in Xh:
                mats[n].spmm_host(Xh[(n, N)], Yh[(n, N)], stream=sh)
        dt_sync = _max_over_ranks(time.perf_counter() - t1, ws)
        e2e = {"value": round(ws * e2e_bytes * reps / dt / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "blocking_calls_value": round(ws * e2e_bytes * reps / dt_sync / 1e9, 1),
               "note": "16 bsp_spmm_host_async calls per step (4 layers x N=1,2,8,16) from pinned host X "
                       "to pinned host Y (H2D, kernel, D2H each), the layers on two streams, synchronised once "
                       "per step, host wall clock; blocking_calls_value: bsp_spmm_host on one stream, "
                       "synchronising after every call"}

    prefill = None
    if not args.no_prefill:
        _progress("prefill leg")
        prefill = run_prefill_leg(bsp, torch, dev, stream, ws)

    union = None
    if not args.no_union:
        _progress("union leg")
        union = run_union_leg(bsp, torch, dev, stream, ws)

    sweep = None
    if not args.no_sweep:
        _progress("sweep leg")
        sweep = run_sweep_leg(bsp, torch, dev, stream, ws)

    int8 = None
    if not args.no_int8:
        _progress("int8 leg")
        int8 = run_int8_leg(bsp, torch, dev, stream, ws)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = time_oracle(Ws, xs, relu, bpc, stor, target_s=10.0)
        cpu.update(time_oracle_extra(Ws, xs, relu, bpc, stor))

    d = by_kernel[dom]
    dach = d["bytes"] / (d["ms"] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dach, 1), "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": round(dach / peak, 4),
                "algorithmic_bytes_per_launch": round(d["bytes"] / d["launches"]),
                "launches_per_step": d["launches"], "share_of_step_time": round(d["ms"] / launch_ms, 4),
                "traffic": traffic,
                "by_kernel": {n: {"launches_per_step": e["launches"],
                                  "achieved": round(e["bytes"] / (e["ms"] * 1e-3) / 1e9, 1),
                                  "frac": round(e["bytes"] / (e["ms"] * 1e-3) / 1e9 / peak, 4),
                                  "share_of_step_time": round(e["ms"] / launch_ms, 4),
                                  "traffic": traffic_kernels.get(n, {}).get("dram_bytes_per_launch")}
                              for n, e in by_kernel.items()},
                "step": {"kernels": STEP_KERNELS, "achieved": round(achieved, 1),
                         "frac": round(achieved / peak, 4),
                         "algorithmic_bytes_per_launch": round(step_bytes / n_calls)}}
    # flat scalars beside the nested records (readers that keep only the
    # scalar fields of each object still see every headline figure)
    for key, b in breakdown.items():
        if key.startswith("N="):
            roofline[f"frac_hbm_N{key[2:]}"] = b["frac_hbm"]
            roofline[f"GBps_N{key[2:]}"] = b["GBps"]
    roofline["spmspv_fc2_GBps"] = breakdown["spmspv_fc2"]["GBps"]
    roofline["spmspv_fc2_us"] = breakdown["spmspv_fc2"]["us"]
    roofline["spmspv_fc2_speedup_vs_spmm_n1"] = breakdown["spmspv_fc2"]["speedup_vs_spmm_n1"]
    for n, e in roofline["by_kernel"].items():
        roofline[f"{n}_frac"] = e["frac"]
        roofline[f"{n}_share"] = e["share_of_step_time"]
    roofline["step_achieved"] = roofline["step"]["achieved"]
    roofline["step_frac"] = roofline["step"]["frac"]
    if sweep:
        for sk, row in sweep["points"].items():
            for N in SWEEP_NS:
                roofline[f"sweep_{sk.replace('=', '').replace('.', '')}_N{N}_frac"] = row[f"N={N}"]["frac_hbm"]
            roofline[f"sweep_{sk.replace('=', '').replace('.', '')}_N1_us"] = row["N=1"]["us"]
    if int8:
        best = 0.0
        for pk, row in int8["points"].items():
            tag = pk.replace(" s=", "_s").replace(".", "")
            for N in INT8_NS:
                roofline[f"{tag}_N{N}_GBps"] = row[f"N={N}"]["GBps"]
                best = max(best, row[f"N={N}"]["frac_hbm"])
        roofline["int8_best_frac"] = best
    if union:
        for lk in ("W4A4", "W4A4_reordered", "W8A8"):
            for N in UNION_NS:
                roofline[f"union_{lk}_N{N}_frac"] = union[lk]["points"][f"N={N}"]["frac_hbm"]
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
                "data": "synthetic (seeded numpy: N(0,0.02) weights, magnitude 50% mask, N(0,1) X)",
                "config": _config(), "frac_hbm": round(value / ws / peak, 4),
                "breakdown": breakdown, "prefill": prefill, "union_ie_bme": union,
                "sparsity_sweep": sweep, "int8": int8,
                "roofline": roofline,
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps * sum(LAUNCHES_PER_CALL[step_kernel(k)] for k, _ in calls),
                "clocks": clk}
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


UNION_NS = (1, 8, 16)


def run_union_leg(bsp, torch, dev, stream, ws, steps=20):
    """IE-BME union-bitmap product (UnionSparse), W4A4 and W8A8, on the four
    OPT-13B projections at 50% (i.i.d. Bernoulli masks, nonzeros uniform
    over the b-bit range), N = 1, 8, 16.  GB/s of the algorithmic bytes
    (union storage + int8 X + int32 Y) with the four layers rotating through
    L2 (178 MB of W4 storage, 340 MB of W8); also the storage against dense
    b-bit bytes and the page's PMR.  W4A4 is measured twice: as encoded and
    with bitmap-aware row reordering (encode time, union entries saved)."""
    peak, peak_kind = _peaks()
    out = {"unit": "GB/s", "peak": peak, "peak_kind": peak_kind}
    for bits, reorder in ((4, False), (4, True), (8, False)):
        mats, X, Y, bpc = {}, {}, {}, {}
        stor_total = dense_total = payload_total = values_total = 0
        enc_s = 0.0
        for li, (name, M, K) in enumerate(LAYERS):
            W = synth.weights_int(M, K, bits, 0.5, synth.seed_for(6, 10 * bits + li), exact=False)
            Wd = torch.from_numpy(W).to(dev)
            del W
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            A = bsp.UnionMatrix(Wd, bits, reorder=reorder)
            torch.cuda.synchronize()
            enc_s += time.perf_counter() - t0
            del Wd
            info = A.info()
            values_total += info["total_values"]
            stor = A.storage_bytes()
            stor_total += stor
            dense_total += M * K * bits // 8
            payload_total += info["nnz"] * bits / 8
            mats[name] = A
            for N in UNION_NS:
                X[(name, N)] = torch.from_numpy(synth.activations_int(N, K, bits, synth.seed_for(6, N))).to(dev)
                Y[(name, N)] = torch.empty((N, M), dtype=torch.int32, device=dev)
                bpc[(name, N)] = stor + K * N + 4 * M * N
        leg = {"storage_bytes": stor_total, "dense_bytes": dense_total,
               "compression_ratio": round(dense_total / stor_total, 4),
               "pmr": round(payload_total / (stor_total - payload_total), 4),
               "stored_values": values_total, "encode_seconds": round(enc_s, 3), "points": {}}
        for N in UNION_NS:
            def rnd():
                for name, _, _ in LAYERS:
                    mats[name].spmm(X[(name, N)], out=Y[(name, N)], stream=stream)
            for _ in range(3):
                rnd()
            torch.cuda.synchronize()
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(steps):
                rnd()
            e0.record(stream)
            torch.cuda.synchronize()
            ms = _max_over_ranks(s0.elapsed_time(e0) / steps, ws)
            b = sum(bpc[(name, N)] for name, _, _ in LAYERS)
            gbps = b / (ms * 1e-3) / 1e9
            leg["points"][f"N={N}"] = {"us_per_round": round(ms * 1e3, 2), "GBps": round(gbps, 1),
                                       "frac_hbm": round(gbps / peak, 4)}
        for A in mats.values():
            A.check()
            A.close()
        out[f"W{bits}A{bits}" + ("_reordered" if reorder else "")] = leg
    return out


def run_int8_leg(bsp, torch, dev, stream, ws, steps=20):
    """INT8 bitmap SpMM (int8 W and X, exact int32 accumulation) on the
    11008 x 4096 and 4096 x 11008 layers at 50% and 60%, N = 1, 8, 16.
    Each configuration is encoded into enough copies to hold three times L2,
    and the calls rotate over them, so every call reads its weight from HBM;
    GB/s of the algorithmic bytes (storage + K*N + 4*M*N) per call."""
    peak, peak_kind = _peaks()
    out = {"unit": "GB/s", "peak": peak, "peak_kind": peak_kind, "points": {}}
    for li, (name, M, K) in enumerate(INT8_LAYERS):
        for s in INT8_SPARSITY:
            W, X, _ = int8_inputs(li, s)
            Wd = torch.from_numpy(W).to(dev)
            first = bsp.BitmapMatrix(Wd)
            stor = first.storage_bytes()
            copies = max(2, -(-3 * L2_BYTES // stor))
            mats = [first] + [bsp.BitmapMatrix(Wd) for _ in range(copies - 1)]
            del Wd
            torch.cuda.synchronize()
            row = {"storage_bytes": stor, "compression_ratio": round(M * K / stor, 4), "copies": copies}
            for N in INT8_NS:
                _progress(f"int8 {name} s={s} N={N}")
                Xd = torch.from_numpy(X[:N].copy()).to(dev)
                Y = torch.empty((N, M), dtype=torch.int32, device=dev)

                def rnd():
                    for A in mats:
                        A.spmm(Xd, out=Y, stream=stream)
                for _ in range(3):
                    rnd()
                torch.cuda.synchronize()
                s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record(stream)
                for _ in range(steps):
                    rnd()
                e0.record(stream)
                torch.cuda.synchronize()
                us = _max_over_ranks(s0.elapsed_time(e0) / (steps * copies), ws) * 1e3
                gbps = (stor + K * N + 4 * M * N) / (us * 1e-6) / 1e9
                row[f"N={N}"] = {"us": round(us, 2), "GBps": round(gbps, 1), "frac_hbm": round(gbps / peak, 4)}
            for A in mats:
                A.check()
                A.close()
            out["points"][f"{name} s={s:.1f}"] = row
    return out


def run_prefill_leg(bsp, torch, dev, stream, ws, reps=5):
    """Prefill TFLOP/s (tcgen05 kernel) on the Llama-2-70B FFN shapes.

    Executed flops = 2*M*K*N (the decoded tile is multiplied densely, zeros
    included, as on the pages); useful flops = 2*NNZ*N.  Each (layer, N) is
    timed over `reps` calls with CUDA events after 3 warm-up calls; the
    encoded weight (264 MB) is larger than L2."""
    peak, peak_kind = _tensor_peak()
    out = {"unit": "TFLOP/s", "peak": peak, "peak_kind": peak_kind, "points": {}}
    best = None
    for name, M, K in PREFILL_LAYERS:
        W = prefill_weights(name, M, K)
        nnz = int(np.count_nonzero(W))
        A = bsp.BitmapMatrix(torch.from_numpy(W.view(np.float16)).to(dev))
        del W
        for N in PREFILL_NS:
            X = torch.from_numpy(prefill_acts(N, K).view(np.float16)).to(dev)
            Y = torch.empty((N, M), dtype=torch.float16, device=dev)
            for _ in range(3):
                A.spmm(X, out=Y, stream=stream)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s.record(stream)
            for _ in range(reps):
                A.spmm(X, out=Y, stream=stream)
            e.record(stream)
            torch.cuda.synchronize()
            ms = _max_over_ranks(s.elapsed_time(e) / reps, ws)
            tf = 2.0 * M * K * N / (ms * 1e-3) / 1e12
            out["points"][f"{name} {M}x{K} N={N}"] = {
                "ms": round(ms, 4), "TFLOPs": round(tf, 1), "frac": round(tf / peak, 4),
                "useful_TFLOPs": round(2.0 * nnz * N / (ms * 1e-3) / 1e12, 1)}
            out[f"{name}_N{N}_TFLOPs"] = round(tf, 1)
            out[f"{name}_N{N}_frac"] = round(tf / peak, 4)
            if best is None or tf > best[0]:
                best = (tf, f"{name} N={N}")
            del X, Y
        A.check()
        A.close()
    out["best"] = {"TFLOPs": round(best[0], 1), "frac": round(best[0] / peak, 4), "at": best[1]}
    out["best_TFLOPs"] = out["best"]["TFLOPs"]
    out["best_frac"] = out["best"]["frac"]
    out["best_at"] = best[1]
    return out


SWEEP_SHAPE = (8192, 8192)
SWEEP_SPARSITY = (0.3, 0.4, 0.5, 0.6, 0.7)
SWEEP_NS = (1, 4, 8, 16)
L2_BYTES = 129 * 10**6


def sweep_closed_form(M, K, nnz):
    """Storage of an M x K fp16 layer (M, K multiples of 64) holding nnz
    stored values, written from the format's parts: 2 bytes per value, one
    8-byte bitmap per 8 x 8 tile, one 4-byte offset per 64 x 64 group plus
    the end offset."""
    return 2 * nnz + 8 * (M * K // 64) + 4 * (M * K // 4096 + 1)


def sweep_nominal_bytes(M, K, s):
    """The same closed form at the nominal count of kept values, M*K -
    round(s*M*K); a few N(0, 0.02) draws round to an fp16 zero, which the
    format does not store, so the measured storage is a little lower."""
    return sweep_closed_form(M, K, M * K - round(s * M * K))


def run_sweep_leg(bsp, torch, dev, stream, ws, steps=20):
    """Sparsity sweep of the decode product on a square 8192 x 8192 fp16
    layer: uniform exact-count masks at 30-70%, N(0, 0.02) values, N(0, 1)
    activations, N = 1, 4, 8, 16.  Per sparsity: the library's storage
    against the closed form, CR = dense fp16 bytes / storage; per point the
    GB/s of the algorithmic bytes (storage + 2KN + 2MN) and its fraction of
    the HBM peak.  The layer is encoded into enough separate copies that the
    copies together hold at least three times L2 and the calls rotate over
    them, so every call reads its weight from HBM."""
    peak, peak_kind = _peaks()
    M, K = SWEEP_SHAPE
    out = {"shape": f"{M}x{K} fp16", "unit": "GB/s", "peak": peak, "peak_kind": peak_kind, "points": {}}
    for s in SWEEP_SPARSITY:
        W = sweep_weights(s)
        nnz = int(np.count_nonzero(W))
        Wd = torch.from_numpy(W.view(np.float16)).to(dev)
        del W
        first = bsp.BitmapMatrix(Wd)
        stor = first.storage_bytes()
        copies = max(2, -(-3 * L2_BYTES // stor))
        mats = [first] + [bsp.BitmapMatrix(Wd) for _ in range(copies - 1)]
        del Wd
        torch.cuda.synchronize()
        closed = sweep_closed_form(M, K, nnz)
        if stor != closed:
            raise RuntimeError(f"storage {stor} != closed form {closed} at s={s}")
        row = {"nnz": nnz, "storage_bytes": stor, "closed_form_bytes": closed,
               "nominal_closed_form_bytes": sweep_nominal_bytes(M, K, s),
               "compression_ratio": round(2 * M * K / stor, 4), "copies": copies}
        for N in SWEEP_NS:
            X = torch.from_numpy(sweep_acts(N).view(np.float16)).to(dev)
            Y = torch.empty((N, M), dtype=torch.float16, device=dev)

            def rnd():
                for A in mats:
                    A.spmm(X, out=Y, stream=stream)
            for _ in range(3):
                rnd()
            torch.cuda.synchronize()
            s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(steps):
                rnd()
            e0.record(stream)
            torch.cuda.synchronize()
            us = _max_over_ranks(s0.elapsed_time(e0) / (steps * copies), ws) * 1e3
            gbps = (stor + 2 * K * N + 2 * M * N) / (us * 1e-6) / 1e9
            row[f"N={N}"] = {"us": round(us, 2), "GBps": round(gbps, 1), "frac_hbm": round(gbps / peak, 4)}
        for A in mats:
            A.check()
            A.close()
        out["points"][f"s={s:.1f}"] = row
    return out


def _kernel_hash():
    """Hash of the kernel sources the decode step launches (the stored DRAM
    traffic is used only while they are unchanged)."""
    import hashlib
    h = hashlib.sha256()
    for name in STEP_SOURCES:
        with open(os.path.join(ROOT, "bitmap_encoded_unstructured_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-union", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-int8", action="store_true")
    ap.add_argument("--case", default=None,
                    help="LAYER:N, one configuration only (N=0: spMspV; int8_11008x4096 / int8_4096x11008: "
                         "the int8 layers at 50%%), for profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    from bitmap_encoded_unstructured_gb300.build import build_library
    build_library()
    if args.case:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
