"""Sharded receiver (the all-to-all of §3.3 of the LoCo paper) without a GPU:
the shard map of loco_shard_range, and the exchange and the 16-bit parameter
all-gather of bit_gradient_compression_gb300.sharded on 2 and 3 gloo ranks
(CPU tensors): every rank must receive exactly the block-aligned slices of all
ranks' packed buffers that belong to its shard."""
import ctypes
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import build
    build.build()
    from bit_gradient_compression_gb300 import loco
    return loco


CASES = [  # (n, bits, block)
    (5 * 1024 + 77, 4, 256),      # ragged last shard
    (3 * 4 * 64 * 7, 8, 64),      # whole units, equal shards for W = 3
    (100, 4, 64),                 # fewer units than ranks: empty shards
    (1, 8, 128),
    (4 * 128 * 11 + 128 + 3, 8, 128),
]


def test_shard_map_properties(L):
    for n in [0, 1, 63, 64, 255, 256, 1023, 1024, 1025, 4095, 4096, 4097, 10 ** 6 + 17, 6_738_415_616]:
        for block in (64, 128, 256):
            U = 4 * block
            nu = -(-n // U)
            for W in range(1, 17):
                rs = [L.loco_shard_range(n, block, W, j) for j in range(W)]
                assert rs[0][0] == 0 and rs[-1][1] == n
                for (l0, h0), (l1, h1) in zip(rs, rs[1:]):
                    assert h0 == l1                                    # contiguous, in rank order
                for lo, hi in rs:
                    assert 0 <= lo <= hi <= n
                    assert lo % U == 0 or lo == n                      # starts on a unit boundary
                    assert hi % U == 0 or hi == n
                units = [-(-(hi - lo) // U) for lo, hi in rs]
                assert sum(units) == nu
                assert max(units) - min(units) <= 1                    # balanced to one unit
                assert sum(u > 0 for u in units) == min(W, nu)
                # codes and steps of every non-empty shard start 16-byte aligned in a rank's buffers
                for lo, hi in rs:
                    for bits in ((4, 8) if hi > lo else ()):
                        assert (lo * bits // 8) % 16 == 0 and (lo // block * 4) % 16 == 0


def test_shard_map_errors(L):
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    f = L.lib.loco_shard_range
    assert f(100, 256, 4, 0, None, ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(100, 256, 4, 4, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(100, 256, 4, -1, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(100, 256, 0, 0, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(-1, 256, 2, 0, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(L.LOCO_MAX_N + 1, 256, 2, 0, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_INVALID_ARG
    assert f(100, 32, 2, 0, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_UNSUPPORTED
    assert f(100, 256, 17, 0, ctypes.byref(lo), ctypes.byref(hi)) == L.LOCO_ERR_UNSUPPORTED


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_buffers(rank, n, bits, block):
    """Rank r's packed bucket as it would leave loco_compress (random bytes and steps)."""
    import torch
    from bit_gradient_compression_gb300 import loco as L
    from bit_gradient_compression_gb300.sharded import scales_capacity
    g = torch.Generator().manual_seed(1000 + 17 * rank + n)
    codes = torch.randint(0, 256, (L.loco_code_bytes(n, bits, block),), dtype=torch.uint8, generator=g)
    scales = torch.rand(scales_capacity(n, block), generator=g)
    return codes, scales


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from bit_gradient_compression_gb300.sharded import ShardedReceiver
    out = []
    try:
        for n, bits, block in CASES:
            rx = ShardedReceiver(n, bits, block)
            codes, scales = _rank_buffers(rank, n, bits, block)
            rx.exchange(codes, scales)
            got_c, got_s = rx.slices()
            ok = len(got_c) == world and len(got_s) == world
            nb_me = -(-rx.n_shard // block)
            c0, s0 = rx.lo * bits // 8, rx.lo // block
            for r in range(world):
                rc, rs = _rank_buffers(r, n, bits, block)
                ok &= torch.equal(got_c[r], rc[c0:c0 + got_c[r].numel()])
                ok &= got_c[r].numel() == L_code_bytes(rx.n_shard, bits, block)
                ok &= torch.equal(got_s[r][:nb_me], rs[s0:s0 + nb_me])
                ok &= got_s[r].numel() % 4 == 0                  # every slot a whole number of 16-byte pieces
            # 16-bit parameter all-gather: rank j's shard filled with a pattern of its own
            pat = lambda j, m: (torch.arange(m, dtype=torch.int32) * 7 + 1000 * j).to(torch.int16)
            rx.bf16_send[:rx.n_shard].copy_(pat(rank, rx.n_shard))
            full = rx.unpad(rx.gather_params_bf16())
            want = torch.cat([pat(j, h - l) for j, (l, h) in enumerate(rx.ranges)])
            ok &= full.numel() == n and torch.equal(full, want)
            out.append((n, bits, block, bool(ok)))
        q.put((rank, out, None))
    except Exception as ex:  # report, then let the parent fail the test
        q.put((rank, out, repr(ex)))
    dist.barrier()
    dist.destroy_process_group()


def L_code_bytes(n, bits, block):
    return -(-n // block) * block * bits // 8 if n > 0 else 0


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_and_gather_gloo(L, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in ps:
        p.start()
    res = [q.get(timeout=300) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, err in res:
        assert err is None, f"rank {rank}: {err}"
        assert len(out) == len(CASES)
        for n, bits, block, ok in out:
            assert ok, f"rank {rank}: n={n} bits={bits} block={block}"
