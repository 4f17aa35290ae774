"""The N > 1 host logic of bench.py on CPU ranks (gloo, world size 2).

The hot path shards by sequence with no data exchange: each rank runs its
own batch; only the timings meet, as a max over ranks.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        q.put((rank, bench.max_over_ranks(mine, "cpu"), bench.rank_seed(rank)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_seeds():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, vals, seed in got:
        assert vals == [2.0, 5.0, 0.5]
    assert len({seed for _, _, seed in got}) == world  # independent batches


def test_tokens_scale_with_ranks():
    assert bench.decoded_tokens_per_step(4) == 4 * bench.decoded_tokens_per_step(1)
    D = bench.DECODE_CFG
    assert bench.decoded_tokens_per_step(1) == len(D["windows"]) * D["B"] * D["steps"] * D["layers"]
