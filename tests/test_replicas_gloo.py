"""bench.py's multi-GPU mode runs independent replicas (the path has no
exchange step).  Check its host-side logic with two gloo ranks on the CPU:
each rank gets its own workload, the step time is the max over ranks and
the token count the sum."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        w = bench.replica_workload("decode", r)
        t_max = bench.reduce_over_ranks(1.5 * (r + 1), "max", dist, "cpu")
        tokens = bench.reduce_over_ranks(w.num_tokens, "sum", dist, "cpu")
        out[r] = (r, wsz, local, t_max, tokens, int(w.context_lens.sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        rank, wsz, local, t_max, tokens, ctx = res[r]
        assert (rank, wsz, local) == (r, world, r)
        assert t_max == 3.0                   # max over ranks of 1.5 * (rank + 1)
        assert tokens == 2 * 256              # both replicas' tokens
    assert res[0][5] != res[1][5]             # different seeds -> different contexts
