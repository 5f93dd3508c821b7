"""The replicas path of bench.py across processes, on CPU with gloo (world size 2).

Decode has no exchange step: N GPUs run N independent replicas and the whole-job
value is the bytes of all ranks over the slowest rank's step time. This checks the
cross-rank reduction the benchmark uses, with two real processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    kv = 1_000_000_000
    ms = [2.0, 3.0][rank]        # rank 1 is the slowest
    e2e = [5.0, 4.0][rank]
    out = bench.aggregate_over_ranks(kv, ms, e2e, world, torch.device("cpu"))
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_value_uses_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank in (0, 1):
        value, e2e, ms_max, e2e_max = res[rank]
        assert ms_max == 3.0 and e2e_max == 5.0
        assert value == pytest.approx(2 * 1e9 / 3e-3 / 1e9)
        assert e2e == pytest.approx(2 * 1e9 / 5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import bench
    v, e, m, em = bench.aggregate_over_ranks(10**9, 4.0, 8.0, 1, torch.device("cpu"))
    assert (m, em) == (4.0, 8.0) and v == pytest.approx(250.0) and e == pytest.approx(125.0)
