"""The multi-GPU mode of bench.py is replicas only: every rank runs its own layer,
no collective touches the data path, and the job's step time is the maximum over
ranks. Checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slow replica
        ms = bench.reduce_max(local_ms)
        results[rank] = (w, r, local, ms, bench.job_tokens_per_s(w, 65536, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][:3] == (2, 0, 0) and res[1][:3] == (2, 1, 1)
    for r in (0, 1):
        assert res[r][3] == 15.0                       # max over ranks, seen by both
        assert res[r][4] == pytest.approx(2 * 65536 / 0.015)


def test_single_process_needs_no_process_group():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_tokens_per_s(1, 65536, 40.0) == pytest.approx(65536 / 0.040)
