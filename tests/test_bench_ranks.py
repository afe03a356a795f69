"""bench.py's multi-rank aggregation on two gloo ranks (CPU): every rank runs an
independent replica, the timing is the slowest rank's, and the value counts the
units of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([10.0 + rank, 50.0 - 20.0 * rank], "cpu")
    q.put((rank, got, bench.whole_job_value(10 ** 9, world, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value in res:
        assert got == [11.0, 50.0]
        assert value == pytest.approx(2 * 1e9 / 11e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.whole_job_value(2 * 10 ** 9, 1, 1000.0) == pytest.approx(2.0)


def test_workload_overrides():
    import bench
    w = bench.workload("llama2-7b")
    assert (w.name, w.n, w.bits, w.block, w.W) == ("llama2-7b-bf16", 6738415616, 4, 256, 8)
    assert bench.workload("llama2-7b", 4, 256, 8) == w          # overrides equal to the defaults change nothing
    o = bench.workload("flat:30", bits=8, ranks=16)
    assert (o.n, o.bits, o.block, o.W) == (1 << 30, 8, 256, 16)
    assert o.name == "flat-bf16-2^30[bits=8,W=16]"                # a changed config never matches stored counters
    assert bench.kernel_bytes(1 << 10, 2, 8, 256, 16)["decode_reduce"] == 16 * (1024 + 16) + 4096
