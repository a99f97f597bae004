"""The bench's multi-process path on the CPU: two gloo ranks (replicas), the
time taken as the maximum over ranks and the whole-job tokens/s computed from
it, and torchrun's environment read back.  No GPU is involved."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist() == (rank, world, rank)
        ms, value = bench.whole_job(times[rank], 10, 1000, world,
                                    lambda v: bench._reduce_max(dist, torch, v, torch.device("cpu")))
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    times = [50.0, 80.0]  # ms for 10 steps on each rank
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == 8.0                        # slowest rank: 80 ms / 10 steps
        assert abs(value - 2 * 1000 / 8e-3) < 1e-6  # both ranks' tokens over that time


def test_single_process_defaults():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench._dist() == (0, 1, 0)
    ms, value = bench.whole_job(30.0, 3, 500, 1, lambda v: v)
    assert ms == 10.0 and value == 500 / 10e-3
