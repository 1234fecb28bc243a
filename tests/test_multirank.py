"""Host logic of bench.py's multi-GPU mode on CPU: two gloo ranks, barrier and max-over-ranks
timing (each GPU runs its own replica; the data path has no collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench._barrier(world)
    t = bench._max_over_ranks(10.0 + 5.0 * rank, world)        # each rank's own timing
    with open(os.path.join(out_dir, "rank%d" % rank), "w") as f:
        f.write(repr(t))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [float(open(os.path.join(tmp_path, "rank%d" % r)).read()) for r in range(world)]
    assert got == [15.0, 15.0]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench._max_over_ranks(3.25, 1) == 3.25
    bench._barrier(1)
