"""Host-side logic of `bench.py --gpus N` (independent replicas, one per rank): the timed region
is bracketed by barriers, and the job time is the maximum over ranks.  Run as two gloo ranks on
the CPU; no GPU involved."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, l = bench.dist_setup()
    assert (w, r, l) == (world, rank, rank)
    bench.barrier(w)
    mine = 10.0 + 5.0 * rank                      # per-rank elapsed ms
    out[rank] = bench.max_over_ranks(mine, w, torch.device("cpu"))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_max_over_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench.barrier(1)
