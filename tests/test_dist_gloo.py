"""Cross-rank logic of the sharded step, on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tree_causal_verification_gb300.dist import job_throughput, max_over_ranks, shard_sequences


def test_shard_sequences_cover_each_sequence_once():
    for batch in (0, 1, 5, 16, 64, 67):
        for world in (1, 2, 3, 4, 8):
            owned = [i for r in range(world) for i in shard_sequences(batch, r, world)]
            assert owned == list(range(batch))
            sizes = [len(shard_sequences(batch, r, world)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_sequences(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r processed 10*(r+1) units in (r+1) seconds: the job took the
        # slowest rank's 2 s and processed 30 units -> 15 units/s.
        tput = job_throughput(10.0 * (rank + 1), float(rank + 1))
        mx = max_over_ranks(float(rank) * 3.0)
        mine = list(shard_sequences(64, rank, world))
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        out[rank] = (tput, mx, sorted(sum(gathered, [])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_benchmark():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        tput, mx, allseq = out[r]
        assert tput == pytest.approx(15.0)
        assert mx == pytest.approx(3.0)
        assert allseq == list(range(64))
