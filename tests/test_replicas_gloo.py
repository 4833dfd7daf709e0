"""The N > 1 path of bench.py on CPU: two ranks over gloo, each with its own
seeded batch (replicas only: no decode data crosses ranks); the job's value
is the bytes all ranks moved divided by the slowest rank's step time."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        case = bench.workload("llama8b", rank)
        ab = bench.algorithmic_bytes(case, case.kv_dtype)
        bench.barrier(world)
        ms_local = 0.05 + 0.01 * rank  # rank 1 is the slower one
        ms, total, value = bench.job_throughput(ms_local, ab["total"], world)
        out[rank] = (int(case.seq_lens.sum()), float(ab["total"]), ms, total, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    r0, r1 = out[0], out[1]
    # each rank decodes its own batch (seeded by rank)
    assert r0[0] != r1[0]
    # both ranks agree on the job figures: slowest step, bytes of both batches
    for r in (r0, r1):
        assert r[2] == pytest.approx(0.06)
        assert r[3] == pytest.approx(r0[1] + r1[1])
        assert r[4] == pytest.approx((r0[1] + r1[1]) / 0.06e-3 / 1e9)
