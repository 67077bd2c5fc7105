"""Multi-process path of bench.py (replicas, weak scaling), on CPU with gloo.

`bench.py --gpus N` under torchrun runs N independent replicas; the reported
value is every rank's bytes over the slowest rank's time.  Two gloo ranks on
127.0.0.1 check that reduction (no GPU, no data-path collective).
"""
import os
import socket
import sys

import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        # rank r took 1 + r seconds for 3 GB: the job moved 3 GB per rank in the
        # slowest rank's 1 + (world - 1) seconds
        secs, gbs = bench.replica_rate(1.0 + rank, 3e9, tdist, world)
        out[rank] = (secs, gbs)
    finally:
        tdist.destroy_process_group()


def test_replica_rate_takes_the_slowest_rank_and_all_bytes():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as man:
        out = man.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        got = dict(out)
    for r in range(world):
        secs, gbs = got[r]
        assert secs == 2.0
        assert abs(gbs - 3.0 * world / 2.0) < 1e-12


def test_replica_rate_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_rate(0.5, 2e9, None, 1) == (0.5, 4.0)
