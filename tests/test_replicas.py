"""Replica bookkeeping across ranks, on CPU with the gloo backend (world size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from higher_order_linear_gb300 import replicas


def test_head_range_covers_all_heads_once():
    for BH in (1, 7, 16, 65535):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                b, e = replicas.head_range(BH, r, world)
                assert 0 <= b <= e <= BH
                seen.extend(range(b, e))
            assert seen == list(range(BH))
    with pytest.raises(ValueError):
        replicas.head_range(4, 2, 2)


def test_job_throughput():
    assert replicas.job_throughput(1000, 2, 500.0) == pytest.approx(4000.0)
    with pytest.raises(ValueError):
        replicas.job_throughput(1, 1, 0.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [3.5, 5.25][rank]
        ms = replicas.max_over_ranks(my_ms)
        out[rank] = (ms, replicas.job_throughput(100, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        ctx = mp.get_context("spawn")
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1] == (5.25, pytest.approx(2 * 100 / 5.25e-3))


def test_max_over_ranks_without_process_group():
    assert replicas.max_over_ranks(1.25) == 1.25
