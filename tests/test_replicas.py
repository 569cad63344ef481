"""The multi-rank (N > 1) bench bookkeeping on CPU: two gloo ranks, each a replica with its own
time and work; the job figure must use the slowest rank's time and the work of both."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from gqa_canvas_attention_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [10.0, 25.0][rank]
    units = [3.0e12, 3.0e12][rank]
    q.put((rank, replicas.aggregate(ms, units)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in (0, 1):
        max_ms, units = res[r]
        assert max_ms == 25.0 and units == 6.0e12
    assert replicas.throughput(25.0, 6.0e12) == pytest.approx(2.4e14)


def test_single_process_is_identity():
    assert replicas.aggregate(7.0, 11.0) == (7.0, 11.0)
