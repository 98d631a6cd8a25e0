"""Multi-process path of the benchmark on CPU (gloo, world size 2): each rank is an
independent replica with its own token batch (data parallel, no collective on the
data path); timing takes the slowest rank and throughput counts every rank's tokens."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import oracle
    import synth
    # each replica runs the block on its own seeded batch
    inp = synth.make_custom(6, 32, 4, 2, 16, act="f32", w="f32", seed=100 + rank)
    out = oracle.forward(inp)["out"]
    ms_local = 10.0 * (rank + 1)
    ms = bench.max_over_ranks(ms_local, world)
    gathered = [torch.zeros(6, 32, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(out))
    q.put((rank, ms, bench.job_throughput(world, 6, 5, ms), [g.numpy() for g in gathered]))
    dist.destroy_process_group()


def test_two_replicas_max_timing_and_job_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import oracle
    import synth
    for rank, ms, value, outs in res:
        assert ms == 20.0                     # slowest rank
        assert value == pytest.approx(2 * 6 * 5 / 0.020)
        for r in range(world):                # replica r's result equals a single-process run of its batch
            ref = oracle.forward(synth.make_custom(6, 32, 4, 2, 16, act="f32", w="f32", seed=100 + r))["out"]
            np.testing.assert_array_equal(outs[r], ref)
