"""Multi-rank host logic of bench.py on CPU with the gloo backend (world size 2).

bench.py runs one independent batch per rank (no collective on the data path)
and reduces only its timings with an element-wise max across ranks.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench._dist()
        assert (w, r, local) == (world, rank, rank)
        got = bench.reduce_max([float(rank + 1), 10.0 - rank, 3.5], world)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(",".join(repr(x) for x in got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        vals = [float(x) for x in (tmp_path / f"rank{rank}.txt").read_text().split(",")]
        assert vals == [2.0, 10.0, 3.5]


def test_reduce_max_single_rank_is_identity():
    import bench

    assert bench.reduce_max([1.0, 2.0], 1) == [1.0, 2.0]
