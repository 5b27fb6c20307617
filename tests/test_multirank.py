"""The multi-process path of bench.py on CPU: two gloo ranks agree on the
slowest rank's step time (the only cross-rank step; the decode itself needs
no collective because (sequence, KV head) items are independent)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    got = bench.max_over_ranks(1.5 + rank)
    q.put((rank, got, bench.dist_info()))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2][:2] for r in res] == [(2, 0), (2, 1)]


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
