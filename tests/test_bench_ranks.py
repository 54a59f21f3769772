"""bench.py's multi-rank logic on CPU: two gloo ranks agree on the max time and pass the barrier.
(On GPUs the same functions run over NCCL. There, every rank runs its own replica and there
is no collective on the data path.)"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier(world)
    out[rank] = bench.reduce_max(10.0 + rank * 5.5, world)
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 15.5, 1: 15.5}


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)
