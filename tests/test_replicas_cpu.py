"""The multi-replica bookkeeping of bench.py (one process per GPU, no
data-path collective): two gloo ranks on CPU, each with its own per-rank
time, must both see the maximum (the whole-job time) and pass the barrier
that brackets the timed region."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, values, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist()[:2] == (ws, rank)
        bench._barrier(ws)
        q.put((rank, bench._max_over_ranks(values[rank], ws)))
        bench._barrier(ws)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    ws, port = 2, _free_port()
    values = [1.25, 3.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, values, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = dict(q.get(timeout=10) for _ in range(ws))
    assert got == {0: 3.5, 1: 3.5}
