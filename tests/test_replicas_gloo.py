"""The replica path of the benchmark on CPU: two gloo ranks with different
step times agree on the slowest rank's time and the whole-job rate."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_decode_28_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world_size, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world_size),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world_size)
    try:
        ws, r, lr = replicas.world()
        local_seconds = 0.010 * (rank + 1)  # rank 1 is the slow one
        replicas.barrier(ws)
        slowest = replicas.max_over_ranks(local_seconds, ws)
        rate = replicas.whole_job_rate(581_140_480, ws, slowest)
        q.put((r, lr, ws, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, local, ws, slowest, rate) in enumerate(res):
        assert rank == r and local == r and ws == 2
        assert slowest == pytest.approx(0.020)
        assert rate == pytest.approx(2 * 581_140_480 / 0.020)


def test_single_process_defaults():
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert replicas.world() == (1, 0, 0)
    assert replicas.max_over_ranks(0.5, 1) == 0.5
    assert replicas.whole_job_rate(10, 1, 2.0) == 5.0
