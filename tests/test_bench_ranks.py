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
    agree = (bench.all_ranks_agree(True, "cpu"), bench.all_ranks_agree(rank == 0, "cpu"))
    q.put((rank, got, bench.whole_job_value(10 ** 9, world, got[0]), agree))
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
    for rank, got, value, agree in res:
        assert got == [11.0, 50.0]
        assert value == pytest.approx(2 * 1e9 / 11e-3 / 1e9)
        assert agree == (True, False)      # one rank's "no" is every rank's "no"


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.all_ranks_agree(True, "cpu") is True and bench.all_ranks_agree(False, "cpu") is False
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


def test_algorithmic_bytes_per_element():
    """The roofline numerators: bytes per element of each kernel as the method
    moves them (gradient read, fp32 error read and written, p/8 code bytes and a
    4-byte step per block written; W ranks' codes and steps read by a receiver,
    the fp32 mean written, or param/m/v read and written)."""
    import bench
    n = 1 << 20
    per = lambda d: {k: v / n for k, v in d.items()}
    b = per(bench.kernel_bytes(n, 2, 4, 256, 8))                 # bf16 gradient, 4-bit, block 256, W 8
    assert b["compress"] == pytest.approx(10.515625)
    assert b["decode_reduce"] == pytest.approx(8.125)
    assert b["adam"] == pytest.approx(28.125)
    assert per(bench.kernel_bytes(n, 4, 4, 256, 8))["compress"] == pytest.approx(12.515625)   # fp32 gradient
    assert per(bench.kernel_bytes(n, 2, 8, 128, 8))["compress"] == pytest.approx(11.03125)    # 8-bit, block 128
    e8 = per(bench.kernel_bytes(n, 2, 4, 256, 8, e8=True))      # int8 error: 1 B read + 1 B written + 2 steps/block
    assert e8["compress"] == pytest.approx(2 + 1 + 1 + 0.5 + 12 / 256)
    sgd = per(bench.kernel_bytes(n, 2, 4, 256, 8, optimizer="sgd", bf16_out=True))
    assert sgd["sgd"] == pytest.approx(8 * (0.5 + 4 / 256) + 8 + 2)
    # gradient-equivalent units behind the headline value
    u = bench.grad_units(n, 2, 8)
    assert u == {"compress": 2 * n, "decode_reduce": 16 * n, "adam": 16 * n}


def test_workload_sizes():
    """Parameter counts of the model-shaped buckets, summed from their layouts."""
    import bench
    assert bench.workload("llama2-7b").n == 6_738_415_616
    assert bench.workload("tinyllama").n == 1_100_048_384
    assert bench.workload("mixtral").n == 8 * 3 * 14336 * 4096
    assert bench.workload("flat:26").n == 1 << 26


def test_reference_arm_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON
    line with the keys of the benchmark line, impl = reference, and an e2e
    object that moves no bytes between host and device."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "flat:18", "--steps", "1",
                        "--warmup", "1"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "flat-bf16-2^18" and d["config"]["n_elements"] == 1 << 18
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == pytest.approx(d["value"], rel=1e-3)
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == pytest.approx(d["value"], rel=1e-3)


def test_stored_counters_follow_kernel_code_not_comments():
    """The stored ncu DRAM counters are keyed to each kernel's code: a comment
    edit keeps the key, a code edit changes it, and every timed kernel has
    its own source list."""
    import bench
    base = "int f(int x) {  // doubles x\n  return 2 * x; /* twice */ }\n"
    assert bench.code_of(base) == bench.code_of("int f(int x) { // twice x\n return 2*x;   }".replace("2*x", "2 * x"))
    assert bench.code_of(base) != bench.code_of(base.replace("2 * x", "3 * x"))
    files = {"compress.cu": base, "decode_reduce.cu": base, "adam.cu": base, "sgd.cu": base,
             "receiver_common.cuh": base, "device_common.cuh": base, "loco_internal.h": base}
    h0 = bench.source_hash("adam", read=files.get)
    h1 = bench.source_hash("adam", read=lambda f: files[f] + ("// note\n" if f == "adam.cu" else ""))
    h2 = bench.source_hash("adam", read=lambda f: files[f] + ("int y;\n" if f == "adam.cu" else ""))
    h3 = bench.source_hash("adam", read=lambda f: files[f] + ("int y;\n" if f == "sgd.cu" else ""))
    assert h0 == h1 and h0 != h2 and h0 == h3
    assert set(bench.KERNEL_SOURCES) == {"compress", "decode_reduce", "adam", "sgd"}
