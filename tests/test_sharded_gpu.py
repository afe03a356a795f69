"""Shard-local receiver steps on one GPU (the all-to-all variant of §3.3 of
the LoCo paper): W ranks' packed buckets are cut by loco_shard_range into the
slices the exchange delivers to each shard's owner (the gloo tests check that
the exchange delivers exactly these slices), and the W shard-local decodes and
Adam steps must concatenate bit for bit to the whole-bucket results, which in
turn match the CPU oracle.  A one-rank NCCL group runs the exchange itself."""
import os

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_bits_equal, grad_to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import loco
    torch.cuda.set_device(DEV)
    return loco


def _ranks(L, n, bits, block, W, seed):
    """W ranks' gradients compressed from zero error; scales sized for the exchange."""
    from bit_gradient_compression_gb300 import workloads as wl
    from bit_gradient_compression_gb300.sharded import scales_capacity
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0)
    codes, scales, hosts = [], [], []
    for r in range(W):
        g = wl.fill_flat_normal(torch.empty(n, dtype=torch.bfloat16, device=DEV), wl.seed_for(seed, 1, r),
                                outlier_p=1e-3)
        e = torch.zeros(n, device=DEV)
        c = torch.empty(L.loco_code_bytes(n, bits, block), dtype=torch.uint8, device=DEV)
        s = torch.full((scales_capacity(n, block),), float("nan"), device=DEV)   # padding steps never read
        L.loco_compress(cfg, g, e, 1, c, s)
        codes.append(c)
        scales.append(s)
        hosts.append(grad_to_np(g))
    return cfg, codes, scales


CASES = [(4, 256, 8, 8 * 4 * 256 * 5 + 4 * 256 * 3 + 77), (8, 64, 3, 100_003), (4, 128, 5, 3 * 4 * 128 + 5),
         (8, 256, 2, 1 << 20), (4, 64, 16, 16 * 4 * 64 * 2 + 1)]


@pytest.mark.parametrize("bits,block,W,n", CASES)
def test_shard_local_decode_and_adam_concatenate_to_whole(L, bits, block, W, n):
    cfg, codes, scales = _ranks(L, n, bits, block, W, 300 + W)
    nb = L.loco_num_blocks(n, block)
    mean = torch.empty(n, device=DEV)
    L.loco_decode_reduce(cfg, codes, [s[:nb] for s in scales], n, mean)
    hp = L.make_adam(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.01)
    from bit_gradient_compression_gb300 import workloads as wl
    p0 = wl.fill_uniform(torch.empty(n, device=DEV), 9, -0.05, 0.05)
    pw, mw, vw = p0.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    pbw = torch.empty(n, dtype=torch.int16, device=DEV)
    L.loco_adam_step_bf16(cfg, codes, [s[:nb] for s in scales], n, pw, mw, vw, pbw, hp, 1)
    ps, ms, vs = p0.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    pbs = torch.empty(n, dtype=torch.int16, device=DEV)
    means = torch.full((n,), float("nan"), device=DEV)
    for j in range(W):
        lo, hi = L.loco_shard_range(n, block, W, j)
        if hi == lo:
            continue
        c0, s0 = lo * bits // 8, lo // block
        cb, sb = L.loco_code_bytes(hi - lo, bits, block), -(-(hi - lo) // block)
        sc = [c[c0:c0 + cb] for c in codes]          # what rank j receives from every rank
        ss = [s[s0:s0 + sb] for s in scales]
        L.loco_decode_reduce(cfg, sc, ss, hi - lo, means[lo:hi])
        L.loco_adam_step_bf16(cfg, sc, ss, hi - lo, ps[lo:hi], ms[lo:hi], vs[lo:hi], pbs[lo:hi], hp, 1)
    torch.cuda.synchronize()
    assert_bits_equal(means.cpu().numpy(), mean.cpu().numpy(), "shard means vs whole")
    for a, b, name in ((ps, pw, "param"), (ms, mw, "m"), (vs, vw, "v")):
        assert_bits_equal(a.cpu().numpy(), b.cpu().numpy(), f"shard {name} vs whole")
    assert np.array_equal(pbs.cpu().numpy(), pbw.cpu().numpy())
    om = oracle.decode_reduce([c.cpu().numpy() for c in codes], [s[:nb].cpu().numpy() for s in scales], n,
                              bits=bits, block=block, threads=8)
    assert_bits_equal(mean.cpu().numpy(), om, "whole mean vs oracle")


def test_sharded_step_one_rank_nccl(L, tmp_path):
    """The exchange, the shard-local Adam step and the bf16 all-gather through
    ShardedReceiver on a one-rank NCCL group: the result is the unsharded step."""
    import torch.distributed as dist
    from bit_gradient_compression_gb300.sharded import ShardedReceiver
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    n, bits, block = 4 * 256 * 9 + 13, 4, 256
    cfg, codes, scales = _ranks(L, n, bits, block, 1, 77)
    store = dist.FileStore(str(tmp_path / "store"), 1)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1, device_id=DEV)
    try:
        rx = ShardedReceiver(n, bits, block, device=DEV)
        assert (rx.lo, rx.hi) == (0, n)
        rx.exchange(codes[0], scales[0])
        hp = L.make_adam(lr=1e-3)
        p = torch.linspace(-1, 1, n, device=DEV)
        m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
        rx.adam_step(cfg, rx.shard(p), rx.shard(m), rx.shard(v), hp, 1, bf16=True)
        full = rx.unpad(rx.gather_params_bf16())
        nb = L.loco_num_blocks(n, block)
        p2, m2, v2 = torch.linspace(-1, 1, n, device=DEV), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
        pb2 = torch.empty(n, dtype=torch.int16, device=DEV)
        L.loco_adam_step_bf16(cfg, codes, [scales[0][:nb]], n, p2, m2, v2, pb2, hp, 1)
        torch.cuda.synchronize()
        assert torch.equal(p, p2) and torch.equal(m, m2) and torch.equal(v, v2)
        assert torch.equal(full, pb2)
    finally:
        dist.destroy_process_group()
