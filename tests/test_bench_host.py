"""Host-side logic of bench.py: the multi-rank reduction (gloo, 2 ranks on CPU)
and the JSON contract of the reference arm on a tiny sample."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    r = bench.aggregate(units_per_rank=100.0, seconds=1.0 + rank, world=world)
    out[rank] = (r["value"], r["seconds"])
    dist.destroy_process_group()


def test_aggregate_takes_max_time_over_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    # slowest rank: 2 s; all ranks' units: 200
    for rank in range(world):
        assert res[rank] == (100.0, 2.0)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(50.0, 0.5, 1) == dict(value=100.0, seconds=0.5)


def test_peaks_fallback_or_measured():
    sys.path.insert(0, ROOT)
    import bench

    p = bench.peaks()
    assert p["hbm"] > 1000 and p["bf16"] > 100 and p["source"] in ("measured", "fallback")
