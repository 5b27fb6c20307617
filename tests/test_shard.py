"""Partition by sequence (one GPU per shard) on CPU with two gloo ranks: each
rank takes its contiguous slice of sequences out of one seeded workload, with
the block-table rows and the pages they name; the slices cover every (sequence,
KV head) item exactly once, and the oracle over the slices, put back together,
gives exactly the oracle over the whole batch (items are independent: the
termination rule is per item, so no rank needs another's data)."""
import os
import socket

import numpy as np
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
    import oracle as O
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    res = {}
    for k in (2, 4):
        w = W.config(k, small=True)
        s = W.shard_sequences(w, rank, ws)
        r = O.run_workload(s, eps_mag=1e-2, eps_dir=1e-2, patience=2, threads=1)
        res[k] = dict(lo=s.notes["shard"]["lo"], hi=s.notes["shard"]["hi"], out=r["out"], bu=r["blocks_used"],
                      pool=s.k_cache.shape[0])
    got = [None] * ws
    dist.all_gather_object(got, res)
    q.put((rank, got))
    dist.destroy_process_group()


def test_sequence_shards_gloo():
    import oracle as O
    import workloads as W
    O.build()
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for a, b in zip(res[0][1], res[1][1]):  # every rank received the same shards
        for k in a:
            assert (a[k]["lo"], a[k]["hi"]) == (b[k]["lo"], b[k]["hi"])
            assert np.array_equal(a[k]["bu"], b[k]["bu"]) and np.array_equal(a[k]["out"], b[k]["out"])
    shards = res[0][1]
    for k in (2, 4):
        w = W.config(k, small=True)
        ranges = sorted((sh[k]["lo"], sh[k]["hi"]) for sh in shards)
        assert ranges[0][0] == 0 and ranges[-1][1] == w.batch
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))  # disjoint, no gap
        full = O.run_workload(w, eps_mag=1e-2, eps_dir=1e-2, patience=2, threads=1)
        bu = np.concatenate([sh[k]["bu"] for sh in sorted(shards, key=lambda sh: sh[k]["lo"])])
        out = np.concatenate([sh[k]["out"] for sh in sorted(shards, key=lambda sh: sh[k]["lo"])])
        assert bu.shape == full["blocks_used"].shape == (w.num_items,)
        assert np.array_equal(bu, full["blocks_used"])
        assert np.array_equal(out, full["out"])
        assert sum(sh[k]["pool"] for sh in shards) <= w.k_cache.shape[0]


def test_shard_layout_single_process():
    import workloads as W
    w = W.config(4, small=True)
    for world in (1, 2, 3, 4):
        seen = []
        for r in range(world):
            s = W.shard_sequences(w, r, world)
            lo, hi = W.shard_range(w.batch, r, world)
            seen.extend(range(lo, hi))
            assert s.batch == hi - lo and s.num_items == (hi - lo) * w.num_kv_heads
            for i in range(s.batch):
                n = -(-int(s.seq_lens[i]) // s.page_size)
                # the same K/V rows, through the shard's own table and pool
                np.testing.assert_array_equal(s.k_cache[s.block_table[i, :n]], w.k_cache[w.block_table[lo + i, :n]])
                np.testing.assert_array_equal(s.v_cache[s.block_table[i, :n]], w.v_cache[w.block_table[lo + i, :n]])
            np.testing.assert_array_equal(s.visit_order, w.visit_order[lo:hi])
            np.testing.assert_array_equal(s.q, w.q[lo:hi])
        assert seen == list(range(w.batch))
    with pytest.raises(ValueError):
        W.shard_range(2, 0, 3)
