"""CUDA path vs. CPU oracle, element by element, through the C ABI.

Small and medium buckets (several blocks, ragged tails, every bits/block/dtype
combination, W = 1..16) are compared in full; guard bytes around every output
buffer must survive each call.  The bar is bit-exact: codes and scales are
integer/byte results, and the fp32 error, mean and Adam state are computed in
the same operation order on both sides.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_bits_equal, grad_to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CANARY = 0xA5
GUARD = 64


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import loco
    torch.cuda.set_device(DEV)
    return loco


def wl():
    from bit_gradient_compression_gb300 import workloads
    return workloads


class Guarded:
    """A device buffer with GUARD canary bytes after the part a call may write."""

    def __init__(self, nbytes: int, dtype=torch.uint8):
        self.nbytes = nbytes
        self.raw = torch.full((nbytes + GUARD,), CANARY, dtype=torch.uint8, device=DEV)
        self.dtype = dtype

    def view(self):
        return self.raw[: self.nbytes].view(self.dtype)

    def intact(self) -> bool:
        return bool((self.raw[self.nbytes:] == CANARY).all())


def _grad(n, dtype, seed, outliers=True):
    g = torch.empty(n, dtype=dtype, device=DEV)
    return wl().fill_flat_normal(g, seed, outlier_p=1e-2 if outliers else 0.0)


SIZES = [1, 7, 8, 9, 63, 64, 65, 255, 257, 3 * 2048 + 5, 100_003, 1 << 16]


def _compress_both(L, cfg_kw, n, dtype, steps, seed, fixed_scale=None, grad_fn=None):
    bits, block = cfg_kw["bits"], cfg_kw["block"]
    cfg = L.make_config(fixed_scale=fixed_scale, **cfg_kw)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    e = Guarded(4 * n, torch.float32)
    e.view().zero_()
    codes, scales = Guarded(cb), Guarded(4 * nb, torch.float32)
    e_h = np.zeros(n, dtype=np.float32)
    okw = dict(bits=bits, block=block, beta=cfg_kw["beta"], kappa=cfg_kw["err_scale_mult"],
               reset_period=cfg_kw["reset_period"], fixed_scale=fixed_scale)
    for step in range(1, steps + 1):
        g = grad_fn(step) if grad_fn else _grad(n, dtype, seed + 1000 * step)
        g_h = grad_to_np(g)
        L.loco_compress(cfg, g, e.view(), step, codes.view(), scales.view())
        oc, os_ = oracle.compress(g_h, e_h, step, **okw)
        torch.cuda.synchronize()
        tag = f"n={n} bits={bits} block={block} {dtype} step={step}"
        assert_bits_equal(codes.view().cpu().numpy(), oc, "codes " + tag)
        assert_bits_equal(scales.view().cpu().numpy(), os_, "scales " + tag)
        assert_bits_equal(e.view().cpu().numpy(), e_h, "err " + tag)
        assert e.intact() and codes.intact() and scales.intact(), "guard bytes overwritten " + tag


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_compress_parity_small(L, bits, block, dtype):
    for i, n in enumerate(SIZES):
        _compress_both(L, dict(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=2),
                       n, dtype, 3, 100 * i + bits + block)


@pytest.mark.parametrize("beta", [0.0, 0.5, 1.0, 0.37])
@pytest.mark.parametrize("kappa", [4.0, 6.0])
def test_compress_parity_beta_kappa(L, beta, kappa):
    _compress_both(L, dict(bits=4, block=128, beta=beta, err_scale_mult=kappa, reset_period=3),
                   50_001, torch.bfloat16, 4, 77)


@pytest.mark.parametrize("s", [2.0 ** 19, 2.0 ** 17, 1000.0])
@pytest.mark.parametrize("bits", [4, 8])
def test_compress_parity_fixed_scale(L, s, bits):
    _compress_both(L, dict(bits=bits, block=256, beta=0.9, err_scale_mult=6.0, reset_period=0),
                   20_000 + 3, torch.float32, 3, 91, fixed_scale=s)


def test_compress_zero_and_constant_blocks(L):
    n, block = 64 * 40 + 17, 64

    def gfn(step):
        g = _grad(n, torch.float32, 5 + step)
        g[128:512] = 0            # whole zero blocks
        g[1024:1088] = 3.5e-3     # a constant block
        g[2000:2064] = -7 * 2.0 ** -12
        return g
    _compress_both(L, dict(bits=4, block=block, beta=0.9, err_scale_mult=4.0, reset_period=0), n,
                   torch.float32, 3, 0, grad_fn=gfn)


def test_compress_nonfinite_stays_in_bounds(L):
    """Non-finite input values are outside the contract, but the call must not
    write outside its buffers; finite blocks must still match the oracle."""
    n, bits, block = 4096 + 9, 4, 128
    cfg = L.make_config(bits=bits, block=block)
    g = _grad(n, torch.float32, 3)
    g[130] = float("nan")
    g[700] = float("inf")
    g[1500] = -float("inf")
    e = Guarded(4 * n, torch.float32)
    e.view().zero_()
    codes = Guarded(L.loco_code_bytes(n, bits, block))
    scales = Guarded(4 * L.loco_num_blocks(n, block), torch.float32)
    L.loco_compress(cfg, g, e.view(), 1, codes.view(), scales.view())
    torch.cuda.synchronize()
    assert e.intact() and codes.intact() and scales.intact()
    e_h = np.zeros(n, dtype=np.float32)
    oc, os_ = oracle.compress(grad_to_np(g), e_h, 1, bits=bits, block=block, beta=0.9, kappa=4.0)
    finite_blocks = [b for b in range(L.loco_num_blocks(n, block)) if b not in (1, 5, 11)]
    sc = scales.view().cpu().numpy()
    for b in finite_blocks:
        assert sc[b] == os_[b]


def _random_ranks(L, n, bits, block, W, seed):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    scales = []
    for _ in range(W):
        s = torch.rand(nb, device=DEV, generator=gen) * 1e-3
        s[torch.rand(nb, device=DEV, generator=gen) < 0.05] = 0.0
        scales.append(s)
    return codes, scales


DEC_SIZES = [1, 9, 255, 1000, (1 << 16) + 3]


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 16])
@pytest.mark.parametrize("bits,block", [(4, 256), (4, 64), (8, 128), (8, 256)])
def test_decode_reduce_parity(L, W, bits, block):
    cfg = L.make_config(bits=bits, block=block)
    for i, n in enumerate(DEC_SIZES):
        codes, scales = _random_ranks(L, n, bits, block, W, 1000 * W + i)
        mean = Guarded(4 * n, torch.float32)
        L.loco_decode_reduce(cfg, codes, scales, n, mean.view())
        om = oracle.decode_reduce([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n,
                                  bits=bits, block=block)
        torch.cuda.synchronize()
        assert_bits_equal(mean.view().cpu().numpy(), om, f"mean n={n} W={W}")
        assert mean.intact()


@pytest.mark.parametrize("W", range(1, 17))
@pytest.mark.parametrize("bits,block", [(4, 256), (8, 128)])
def test_decode_reduce_parity_several_tiles_per_warp(L, W, bits, block):
    """2^25 + 37 elements: every warp of the persistent grid walks several
    tiles (its pipeline stages and output tiles wrap around), then the ragged
    tail; every rank has its own codes and steps."""
    n = (1 << 25) + 37
    cfg = L.make_config(bits=bits, block=block)
    codes, scales = _random_ranks(L, n, bits, block, W, 500 + W)
    mean = Guarded(4 * n, torch.float32)
    L.loco_decode_reduce(cfg, codes, scales, n, mean.view())
    om = oracle.decode_reduce([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n,
                              bits=bits, block=block, threads=8)
    torch.cuda.synchronize()
    assert_bits_equal(mean.view().cpu().numpy(), om, f"mean n={n} W={W}")
    assert mean.intact()


@pytest.mark.parametrize("W", [3, 4, 5, 7] + list(range(8, 17)))
def test_decode_reduce_parity_tile_groups(L, W):
    """2^28 + 37 elements, 4-bit codes: at W = 3, 4, 5, 7 and W > 8 the warps of
    the 4-bit decode take groups of 8 consecutive tiles once every warp of the
    resident grid has at least 64 warp tiles (2^28 elements give 108-216 per
    warp); W = 8 keeps the plain order at this size.  Every element is
    compared."""
    n = (1 << 28) + 37
    cfg = L.make_config(bits=4, block=256)
    codes, scales = _random_ranks(L, n, 4, 256, W, 1300 + W)
    mean = Guarded(4 * n, torch.float32)
    L.loco_decode_reduce(cfg, codes, scales, n, mean.view())
    om = oracle.decode_reduce([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n,
                              bits=4, block=256, threads=8)
    torch.cuda.synchronize()
    assert_bits_equal(mean.view().cpu().numpy(), om, f"mean n={n} W={W}")
    assert mean.intact()


@pytest.mark.parametrize("W", [3, 5, 6, 7, 12, 15])
@pytest.mark.parametrize("bits,block", [(4, 64), (8, 128)])
def test_decode_reduce_small_steps_and_signed_zeros(L, W, bits, block):
    """Division by a rank count that is not a power of two: the kernels take a
    two-constant quotient when every step of a block is 0 or >= 2^-77 and the
    IEEE division otherwise.  Blocks whose steps include tiny normal and
    subnormal values (one rank or all), zero steps with negative codes (decoded
    terms -0, so zero sums of either sign) and ordinary steps; mean and the
    fused Adam step bit-exact against the oracle."""
    n = 64 * block + 17
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(70 + W)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    tiny = torch.tensor([2.0 ** -77, 2.0 ** -78, 2.0 ** -100, 2.0 ** -126, 2.0 ** -140, 1e-45], device=DEV)
    scales = []
    for w in range(W):
        sc = torch.rand(nb, device=DEV, generator=gen) * 1e-3
        k = torch.arange(nb, device=DEV)
        sc = torch.where(k % 8 == 1, tiny[k % 6], sc)                          # one tiny step per block...
        sc = torch.where((k % 8 == 2) & (w == W - 1), tiny[(k + w) % 6], sc)   # ...or only the last rank's
        sc = torch.where(k % 8 == 3, torch.zeros_like(sc), sc)                 # zero steps: terms +-0
        sc = torch.where((k % 8 == 4) & (w % 2 == 0), torch.zeros_like(sc), sc)
        scales.append(sc)
    # blocks 5 mod 8: every rank's codes negative with a zero step, so the sum is -0
    bpb = block * bits // 8
    for c, sc in zip(codes, scales):
        cv = c.view(nb, bpb)
        neg = 0x99 if bits == 4 else 0x80
        cv[5::8] = neg
        sc[5::8] = 0.0
    mean = torch.empty(n, device=DEV)
    cfg = L.make_config(bits=bits, block=block)
    L.loco_decode_reduce(cfg, codes, scales, n, mean)
    ch, sh = [c.cpu().numpy() for c in codes], [x.cpu().numpy() for x in scales]
    om = oracle.decode_reduce(ch, sh, n, bits=bits, block=block)
    torch.cuda.synchronize()
    got = mean.cpu().numpy()
    assert_bits_equal(got, om, f"mean W={W}")
    assert np.signbit(got.reshape(-1)[5 * block]) and got.reshape(-1)[5 * block] == 0
    p = wl().fill_uniform(torch.empty(n, device=DEV), 4, -0.1, 0.1)
    m, v = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    ph, mh, vh = p.cpu().numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    hpk = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0)
    L.loco_adam_step(cfg, codes, scales, n, p, m, v, L.make_adam(**hpk), 1)
    oracle.adam_step(ch, sh, n, ph, mh, vh, 1, bits=bits, block=block, **hpk)
    torch.cuda.synchronize()
    for got_t, want, name in ((p, ph, "param"), (m, mh, "m"), (v, vh, "v")):
        assert_bits_equal(got_t.cpu().numpy(), want, f"{name} W={W}")


@pytest.mark.parametrize("W", [1, 3, 8, 16])
@pytest.mark.parametrize("bits,block", [(4, 256), (8, 64)])
@pytest.mark.parametrize("variant", ["adamw", "paper", "plain"])
def test_adam_parity(L, W, bits, block, variant):
    cfg = L.make_config(bits=bits, block=block)
    if variant == "adamw":
        hpk = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, bias_correction=True,
                   eps_inside_sqrt=False)
    elif variant == "paper":
        hpk = dict(lr=3e-4, beta1=0.9, beta2=0.99, eps=1e-10, weight_decay=0.0, bias_correction=False,
                   eps_inside_sqrt=True)
    else:
        hpk = dict(lr=1e-2, beta1=0.0, beta2=0.5, eps=1e-6, weight_decay=0.0, bias_correction=True,
                   eps_inside_sqrt=False)
    hp = L.make_adam(**hpk)
    for i, n in enumerate([7, 1000, (1 << 16) + 5]):
        p = wl().fill_uniform(torch.empty(n, device=DEV), i, -0.05, 0.05)
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        ph, mh, vh = p.cpu().numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        for t in (1, 2, 3):
            codes, scales = _random_ranks(L, n, bits, block, W, 7 * t + i)
            L.loco_adam_step(cfg, codes, scales, n, p, m, v, hp, t)
            oracle.adam_step([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n, ph, mh, vh,
                             t, bits=bits, block=block, **hpk)
            torch.cuda.synchronize()
            assert_bits_equal(p.cpu().numpy(), ph, f"param n={n} t={t}")
            assert_bits_equal(m.cpu().numpy(), mh, f"m n={n} t={t}")
            assert_bits_equal(v.cpu().numpy(), vh, f"v n={n} t={t}")


@pytest.mark.parametrize("eps_inside_sqrt", [False, True])
@pytest.mark.parametrize("W", [1, 2, 5])
def test_adam_parity_zero_and_underflowing_means(L, W, eps_inside_sqrt):
    """Means that are exactly zero (every rank's codes 0 in a block, so m = v = 0
    and the step takes sqrt(0) and 0 / den) and means so small that g*g
    underflows (v = 0 while m != 0), mixed with ordinary blocks, over several
    steps and at sizes that span many tiles plus a ragged tail."""
    bits, block = 4, 64
    cfg = L.make_config(bits=bits, block=block)
    hpk = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8 if not eps_inside_sqrt else 1e-16, weight_decay=0.0,
               bias_correction=True, eps_inside_sqrt=eps_inside_sqrt)
    hp = L.make_adam(**hpk)
    n = 3 * 2048 * 8 + 77
    nb = L.loco_num_blocks(n, block)
    kind = np.arange(nb) % 5            # 0, 1: zero codes; 2: tiny steps; 3, 4: ordinary
    p = wl().fill_uniform(torch.empty(n, device=DEV), 3, -0.05, 0.05)
    m = torch.zeros(n, device=DEV)
    v = torch.zeros(n, device=DEV)
    ph, mh, vh = p.cpu().numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in (1, 2, 3):
        codes, scales = _random_ranks(L, n, bits, block, W, 40 + t)
        for w in range(W):
            c = codes[w].cpu().numpy().reshape(nb, block * bits // 8)
            c[kind <= 1] = 0
            codes[w].copy_(torch.from_numpy(c.reshape(-1)))
            sc = scales[w].cpu().numpy()
            sc[kind == 2] = np.float32(1e-24)
            scales[w].copy_(torch.from_numpy(sc))
        L.loco_adam_step(cfg, codes, scales, n, p, m, v, hp, t)
        oracle.adam_step([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n, ph, mh, vh,
                         t, bits=bits, block=block, **hpk)
        torch.cuda.synchronize()
        assert_bits_equal(p.cpu().numpy(), ph, f"param t={t}")
        assert_bits_equal(m.cpu().numpy(), mh, f"m t={t}")
        assert_bits_equal(v.cpu().numpy(), vh, f"v t={t}")
    assert ((vh == 0) & (mh == 0)).any() and ((vh == 0) & (mh != 0)).any(), "edge cases not reached"


def test_flat_1m_config_full(L):
    """The 1M-element fp32 workload: 4 ranks, 8 steps, 4-bit, block 256,
    beta 0.9 -- every rank's codes, scales and error, and the mean, compared in
    full at every step."""
    W_ = wl()
    w = W_.FLAT_1M
    n, bits, block, W = w.n, w.bits, w.block, w.W
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=512)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    errs = [torch.zeros(n, device=DEV) for _ in range(W)]
    errs_h = [np.zeros(n, np.float32) for _ in range(W)]
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    scales = [torch.empty(nb, device=DEV) for _ in range(W)]
    mean = torch.empty(n, device=DEV)
    for k in range(1, w.steps + 1):
        oc_all, os_all = [], []
        for r in range(W):
            g = w.fill(torch.empty(n, dtype=w.grad_dtype, device=DEV), W_.seed_for(42, k, r))
            L.loco_compress(cfg, g, errs[r], k, codes[r], scales[r])
            oc, os_ = oracle.compress(grad_to_np(g), errs_h[r], k, bits=bits, block=block, beta=0.9, kappa=4.0,
                                      reset_period=512, threads=8)
            oc_all.append(oc)
            os_all.append(os_)
            torch.cuda.synchronize()
            assert_bits_equal(codes[r].cpu().numpy(), oc, f"codes rank {r} step {k}")
            assert_bits_equal(scales[r].cpu().numpy(), os_, f"scales rank {r} step {k}")
            assert_bits_equal(errs[r].cpu().numpy(), errs_h[r], f"err rank {r} step {k}")
        L.loco_decode_reduce(cfg, codes, scales, n, mean)
        om = oracle.decode_reduce(oc_all, os_all, n, bits=bits, block=block, threads=8)
        torch.cuda.synchronize()
        mg = mean.cpu().numpy()
        assert_bits_equal(mg, om, f"mean step {k}")


def test_empty_and_errors(L):
    cfg = L.make_config()
    e = torch.empty(0, device=DEV)
    L.loco_compress(cfg, torch.empty(0, device=DEV), e, 1, torch.empty(0, dtype=torch.uint8, device=DEV),
                    torch.empty(0, device=DEV))
    L.loco_decode_reduce(cfg, [torch.empty(0, dtype=torch.uint8, device=DEV)], [torch.empty(0, device=DEV)], 0,
                         torch.empty(0, device=DEV))
    n = 1000
    g = torch.zeros(n, device=DEV)
    err = torch.zeros(n, device=DEV)
    codes = torch.zeros(L.loco_code_bytes(n, 4, 256), dtype=torch.uint8, device=DEV)
    scales = torch.zeros(L.loco_num_blocks(n, 256), device=DEV)
    with pytest.raises(L.LocoError) as ei:       # host memory
        L.loco_compress(cfg, g.cpu(), err, 1, codes, scales)
    assert ei.value.status == L.LOCO_ERR_INVALID_ARG
    with pytest.raises(L.LocoError) as ei:       # buffer far shorter than n needs
        L.loco_compress(cfg, g, err, 1, codes, scales, n=1 << 40)
    assert ei.value.status == L.LOCO_ERR_INVALID_ARG
    with pytest.raises(L.LocoError) as ei:       # misaligned
        L.loco_compress(cfg, g.data_ptr() + 4, err, 1, codes, scales, n=n - 8, grad_dtype=L.LOCO_F32)
    assert ei.value.status == L.LOCO_ERR_MISALIGNED
    with pytest.raises(L.LocoError) as ei:       # overlapping in/out
        L.loco_compress(cfg, g, g, 1, codes, scales)
    assert ei.value.status == L.LOCO_ERR_INVALID_ARG
    with pytest.raises(L.LocoError) as ei:
        L.loco_decode_reduce(cfg, [codes] * 17, [scales] * 17, n, g)
    assert ei.value.status == L.LOCO_ERR_UNSUPPORTED
    # nothing was launched by the rejected calls, and the stream is still healthy
    torch.cuda.synchronize()
    assert not err.any()


def _compress_e8_both(L, cfg_kw, n, dtype, steps, seed, fixed_scale=None):
    bits, block = cfg_kw["bits"], cfg_kw["block"]
    cfg = L.make_config(fixed_scale=fixed_scale, **cfg_kw)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    qe = Guarded(n, torch.int8)
    qe.view().zero_()
    de = Guarded(4 * nb, torch.float32)
    de.view().zero_()
    codes, scales = Guarded(cb), Guarded(4 * nb, torch.float32)
    qe_h = np.zeros(n, dtype=np.int8)
    de_h = np.zeros(nb, dtype=np.float32)
    okw = dict(bits=bits, block=block, beta=cfg_kw["beta"], kappa=cfg_kw["err_scale_mult"],
               reset_period=cfg_kw["reset_period"], fixed_scale=fixed_scale)
    for step in range(1, steps + 1):
        g = _grad(n, dtype, seed + 1000 * step)
        L.loco_compress_e8(cfg, g, qe.view(), de.view(), step, codes.view(), scales.view())
        oc, os_ = oracle.compress_e8(grad_to_np(g), qe_h, de_h, step, **okw)
        torch.cuda.synchronize()
        tag = f"e8 n={n} bits={bits} block={block} {dtype} step={step}"
        assert_bits_equal(codes.view().cpu().numpy(), oc, "codes " + tag)
        assert_bits_equal(scales.view().cpu().numpy(), os_, "scales " + tag)
        assert_bits_equal(qe.view().cpu().numpy(), qe_h, "err codes " + tag)
        assert_bits_equal(de.view().cpu().numpy(), de_h, "err steps " + tag)
        assert qe.intact() and de.intact() and codes.intact() and scales.intact(), "guard bytes " + tag


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_compress_e8_parity_small(L, bits, block, dtype):
    for i, n in enumerate(SIZES):
        _compress_e8_both(L, dict(bits=bits, block=block, beta=0.1, err_scale_mult=4.0, reset_period=3),
                          n, dtype, 4, 500 + 100 * i + bits + block)


@pytest.mark.parametrize("beta,kappa", [(0.0, 4.0), (0.5, 6.0), (0.9, 4.0), (1.0, 4.0)])
def test_compress_e8_parity_beta_kappa(L, beta, kappa):
    _compress_e8_both(L, dict(bits=4, block=256, beta=beta, err_scale_mult=kappa, reset_period=0),
                      70_001, torch.bfloat16, 4, 9)


@pytest.mark.parametrize("kappa", [0.5, 1.0, 3.0, 2.0 ** -20, 2.0 ** 20])
def test_compress_parity_kappa_powers(L, kappa):
    """kappa a power of two (Delta/kappa taken as an exact product) or not (a division)."""
    _compress_both(L, dict(bits=8, block=64, beta=0.6, err_scale_mult=kappa, reset_period=0),
                   20_011, torch.bfloat16, 3, 21)
    _compress_e8_both(L, dict(bits=4, block=64, beta=0.2, err_scale_mult=kappa, reset_period=0),
                      20_011, torch.bfloat16, 3, 22)


@pytest.mark.parametrize("s", [2.0 ** 19, 2.0 ** 17])
def test_compress_e8_parity_fixed_scale(L, s):
    _compress_e8_both(L, dict(bits=4, block=128, beta=0.5, err_scale_mult=6.0, reset_period=2),
                      30_003, torch.float32, 4, 13, fixed_scale=s)


@pytest.mark.parametrize("bits", [4, 8])
def test_compress_tiny_blocks(L, bits):
    """Blocks whose absmax sits around qmax/FLT_MAX (the inverse step overflows
    fp32 below it), mixed with normal blocks, through both error storages."""
    qmax = 7 if bits == 4 else 127
    thresh = qmax / float(np.finfo(np.float32).max)
    block, nblk = 64, 12
    n = block * nblk - 5
    gh = np.zeros(n, dtype=np.float32)
    rng = np.random.default_rng(bits)
    for b in range(nblk):
        lo, hi = b * block, min((b + 1) * block, n)
        scale = thresh * (0.25, 0.5, 0.999, 1.001, 2.0, 1e30)[b % 6]
        gh[lo:hi] = (rng.uniform(-1, 1, hi - lo) * scale).astype(np.float32)
    g = torch.from_numpy(gh).to(DEV)
    cfg = L.make_config(bits=bits, block=block, beta=0.5)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    e = torch.zeros(n, device=DEV)
    qe = torch.zeros(n, dtype=torch.int8, device=DEV)
    de = torch.zeros(nb, device=DEV)
    c, s = torch.empty(cb, dtype=torch.uint8, device=DEV), torch.empty(nb, device=DEV)
    c8, s8 = torch.empty(cb, dtype=torch.uint8, device=DEV), torch.empty(nb, device=DEV)
    e_h = np.zeros(n, np.float32)
    qe_h, de_h = np.zeros(n, np.int8), np.zeros(nb, np.float32)
    for step in (1, 2):
        L.loco_compress(cfg, g, e, step, c, s)
        L.loco_compress_e8(cfg, g, qe, de, step, c8, s8)
        oc, os_ = oracle.compress(gh, e_h, step, bits=bits, block=block, beta=0.5, kappa=4.0)
        oc8, os8 = oracle.compress_e8(gh, qe_h, de_h, step, bits=bits, block=block, beta=0.5, kappa=4.0)
        torch.cuda.synchronize()
        assert_bits_equal(c.cpu().numpy(), oc, "codes")
        assert_bits_equal(s.cpu().numpy(), os_, "scales")
        assert_bits_equal(e.cpu().numpy(), e_h, "err")
        assert_bits_equal(c8.cpu().numpy(), oc8, "e8 codes")
        assert_bits_equal(s8.cpu().numpy(), os8, "e8 scales")
        assert_bits_equal(qe.cpu().numpy(), qe_h, "e8 err codes")
        assert_bits_equal(de.cpu().numpy(), de_h, "e8 err steps")


@pytest.mark.parametrize("W", [1, 3, 8, 16])
@pytest.mark.parametrize("bits,block", [(4, 256), (8, 64), (4, 128)])
@pytest.mark.parametrize("bf16_out", [False, True])
def test_sgd_parity(L, W, bits, block, bf16_out):
    cfg = L.make_config(bits=bits, block=block)
    for i, n in enumerate([7, 1000, (1 << 16) + 5, 3 * 4096 + 17]):
        p = wl().fill_uniform(torch.empty(n, device=DEV), 40 + i, -0.05, 0.05)
        ph = p.cpu().numpy().copy()
        pb = Guarded(2 * n, torch.int16) if bf16_out else None
        pb_h = np.zeros(n, dtype=np.uint16) if bf16_out else None
        for t in (1, 2, 3):
            codes, scales = _random_ranks(L, n, bits, block, W, 11 * t + i)
            L.loco_sgd_step(cfg, codes, scales, n, p, 3e-3, param_bf16=pb.view() if bf16_out else None)
            oracle.sgd_step([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n, ph,
                            bits=bits, block=block, lr=3e-3, param_bf16=pb_h)
            torch.cuda.synchronize()
            assert_bits_equal(p.cpu().numpy(), ph, f"sgd param n={n} t={t}")
            if bf16_out:
                assert_bits_equal(pb.view().cpu().numpy().view(np.uint16), pb_h, f"sgd bf16 n={n} t={t}")
                assert pb.intact()


@pytest.mark.parametrize("W", range(1, 17))
@pytest.mark.parametrize("bits,block", [(4, 256), (8, 128)])
def test_optimizer_steps_several_tiles_per_cta(L, W, bits, block):
    """2^23 + 37 elements: every CTA of the persistent grid walks several tiles
    (its pipeline stages wrap around, whatever stage count fits at this W),
    then the ragged tail; one Adam(W) step and one SGD step, each rank with its
    own codes and steps."""
    n = (1 << 23) + 37
    cfg = L.make_config(bits=bits, block=block)
    codes, scales = _random_ranks(L, n, bits, block, W, 900 + W)
    codes_h, scales_h = [c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales]
    hpk = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, bias_correction=True,
               eps_inside_sqrt=False)
    p = wl().fill_uniform(torch.empty(n, device=DEV), 5, -0.05, 0.05)
    m = wl().fill_uniform(torch.empty(n, device=DEV), 6, -1e-3, 1e-3)
    v = wl().fill_uniform(torch.empty(n, device=DEV), 7, 0.0, 1e-6)
    ph, mh, vh = p.cpu().numpy().copy(), m.cpu().numpy().copy(), v.cpu().numpy().copy()
    L.loco_adam_step(cfg, codes, scales, n, p, m, v, L.make_adam(**hpk), 3)
    oracle.adam_step(codes_h, scales_h, n, ph, mh, vh, 3, bits=bits, block=block, threads=8, **hpk)
    torch.cuda.synchronize()
    for got_t, want, name in ((p, ph, "param"), (m, mh, "m"), (v, vh, "v")):
        assert_bits_equal(got_t.cpu().numpy(), want, f"adam {name} W={W}")
    q = wl().fill_uniform(torch.empty(n, device=DEV), 8, -0.05, 0.05)
    qh = q.cpu().numpy().copy()
    L.loco_sgd_step(cfg, codes, scales, n, q, 3e-3)
    oracle.sgd_step(codes_h, scales_h, n, qh, bits=bits, block=block, lr=3e-3, threads=8)
    torch.cuda.synchronize()
    assert_bits_equal(q.cpu().numpy(), qh, f"sgd param W={W}")


@pytest.mark.parametrize("W", [1, 8, 13])
@pytest.mark.parametrize("bits,block", [(4, 256), (8, 128)])
def test_adam_bf16_parity(L, W, bits, block):
    cfg = L.make_config(bits=bits, block=block)
    hpk = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, bias_correction=True,
               eps_inside_sqrt=False)
    hp = L.make_adam(**hpk)
    for i, n in enumerate([9, 5000, (1 << 16) + 3]):
        p = wl().fill_uniform(torch.empty(n, device=DEV), 60 + i, -0.05, 0.05)
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        pb = Guarded(2 * n, torch.int16)
        ph, mh, vh = p.cpu().numpy().copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        pb_h = np.zeros(n, dtype=np.uint16)
        for t in (1, 2):
            codes, scales = _random_ranks(L, n, bits, block, W, 5 * t + i)
            L.loco_adam_step_bf16(cfg, codes, scales, n, p, m, v, pb.view(), hp, t)
            oracle.adam_step([c.cpu().numpy() for c in codes], [s.cpu().numpy() for s in scales], n, ph, mh, vh,
                             t, bits=bits, block=block, param_bf16=pb_h, **hpk)
            torch.cuda.synchronize()
            assert_bits_equal(p.cpu().numpy(), ph, f"param n={n} t={t}")
            assert_bits_equal(m.cpu().numpy(), mh, f"m n={n} t={t}")
            assert_bits_equal(v.cpu().numpy(), vh, f"v n={n} t={t}")
            assert_bits_equal(pb.view().cpu().numpy().view(np.uint16), pb_h, f"bf16 n={n} t={t}")
            assert pb.intact()


def test_cuda_graph_capture_replays_the_step(L):
    """The entry points allocate and synchronise nothing, so a whole step
    (compress W ranks, decode-reduce, Adam) can be captured in a CUDA graph and
    replayed; the replay gives the same bits as direct calls."""
    n, bits, block, W = 3 * 4096 + 77, 4, 128, 3
    cfg = L.make_config(bits=bits, block=block, beta=0.9, reset_period=0)
    hp = L.make_adam(lr=1e-3, weight_decay=0.01)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)

    def state():
        gs = [_grad(n, torch.bfloat16, 200 + w) for w in range(W)]
        es = [torch.zeros(n, device=DEV) for _ in range(W)]
        cs = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
        ss = [torch.empty(nb, device=DEV) for _ in range(W)]
        p = wl().fill_uniform(torch.empty(n, device=DEV), 9, -0.1, 0.1)
        return gs, es, cs, ss, p, torch.zeros(n, device=DEV), torch.zeros(n, device=DEV), torch.empty(n, device=DEV)

    def step(st, k, stream=None):
        gs, es, cs, ss, p, m, v, mean = st
        for w in range(W):
            L.loco_compress(cfg, gs[w], es[w], k, cs[w], ss[w], stream=stream)
        L.loco_decode_reduce(cfg, cs, ss, n, mean, stream=stream)
        L.loco_adam_step(cfg, cs, ss, n, p, m, v, hp, k, stream=stream)

    direct = state()
    for k in (1, 2, 3):
        step(direct, k)
    graphed = state()
    step(graphed, 1)                         # first call per kernel does its one-time set-up
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        step(graphed, 2, stream=s)
    g2.replay()
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=s):
        step(graphed, 3, stream=s)
    g3.replay()
    torch.cuda.synchronize()
    for a, b, name in zip(direct, graphed, ("g", "e", "codes", "scales", "p", "m", "v", "mean")):
        if isinstance(a, list):
            for x, y in zip(a, b):
                assert torch.equal(x, y), name
        else:
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), name


@pytest.mark.parametrize("storage", ["fp32", "int8"])
def test_checkpoint_resume(L, storage):
    """The sender's whole state is its error buffer(s) and the step counter: a
    host copy taken after step 3 and restored into fresh buffers continues
    exactly like the uninterrupted run (reset period 4 fires inside the resumed
    part)."""
    n, bits, block = 50_001, 4, 128
    cfg = L.make_config(bits=bits, block=block, beta=0.3, reset_period=4)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    grads = [_grad(n, torch.bfloat16, 900 + k) for k in range(1, 8)]

    def new_state():
        if storage == "fp32":
            return [torch.zeros(n, device=DEV)]
        return [torch.zeros(n, dtype=torch.int8, device=DEV), torch.zeros(nb, device=DEV)]

    def run(state, k, c, s):
        if storage == "fp32":
            L.loco_compress(cfg, grads[k - 1], state[0], k, c, s)
        else:
            L.loco_compress_e8(cfg, grads[k - 1], state[0], state[1], k, c, s)

    full, outs = new_state(), []
    for k in range(1, 8):
        c, s = torch.empty(cb, dtype=torch.uint8, device=DEV), torch.empty(nb, device=DEV)
        run(full, k, c, s)
        outs.append((c, s))
    part = new_state()
    for k in range(1, 4):
        run(part, k, torch.empty(cb, dtype=torch.uint8, device=DEV), torch.empty(nb, device=DEV))
    ckpt = [x.cpu().clone() for x in part]            # checkpoint: plain bytes + step = 3
    del part
    resumed = [x.to(DEV) for x in ckpt]
    for k in range(4, 8):
        c, s = torch.empty(cb, dtype=torch.uint8, device=DEV), torch.empty(nb, device=DEV)
        run(resumed, k, c, s)
        assert torch.equal(c, outs[k - 1][0]) and torch.equal(s, outs[k - 1][1]), k
    for a, b in zip(resumed, full):
        assert torch.equal(a, b)


def test_concurrent_calls_on_independent_streams(L):
    """The kernels keep no state and share no memory beyond their arguments, so
    independent chains of calls running at the same time on four streams give
    the bits of the same chains run one after another."""
    n = 2 * 4096 * 8 + 123
    chains = [dict(bits=4, block=256, W=8, e8=False, opt="adam"), dict(bits=8, block=64, W=5, e8=False, opt="sgd"),
              dict(bits=4, block=128, W=3, e8=True, opt="adam"), dict(bits=8, block=128, W=12, e8=True, opt="sgd")]
    hp = L.make_adam(lr=1e-3, weight_decay=0.01)

    def make(i, c):
        bits, block, W = c["bits"], c["block"], c["W"]
        nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
        st = dict(cfg=L.make_config(bits=bits, block=block, beta=0.2 if c["e8"] else 0.9, reset_period=2),
                  g=[_grad(n, torch.bfloat16, 500 + 20 * i + w) for w in range(W)],
                  cs=[torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)],
                  ss=[torch.empty(nb, device=DEV) for _ in range(W)], mean=torch.empty(n, device=DEV),
                  p=wl().fill_uniform(torch.empty(n, device=DEV), 40 + i, -0.1, 0.1),
                  m=torch.zeros(n, device=DEV), v=torch.zeros(n, device=DEV))
        if c["e8"]:
            st["e"] = [(torch.zeros(n, dtype=torch.int8, device=DEV), torch.zeros(nb, device=DEV)) for _ in range(W)]
        else:
            st["e"] = [torch.zeros(n, device=DEV) for _ in range(W)]
        return st

    def run(c, st, stream):
        for k in (1, 2, 3):
            for w in range(c["W"]):
                if c["e8"]:
                    L.loco_compress_e8(st["cfg"], st["g"][w], st["e"][w][0], st["e"][w][1], k, st["cs"][w], st["ss"][w],
                                       stream=stream)
                else:
                    L.loco_compress(st["cfg"], st["g"][w], st["e"][w], k, st["cs"][w], st["ss"][w], stream=stream)
            L.loco_decode_reduce(st["cfg"], st["cs"], st["ss"], n, st["mean"], stream=stream)
            if c["opt"] == "adam":
                L.loco_adam_step(st["cfg"], st["cs"], st["ss"], n, st["p"], st["m"], st["v"], hp, k, stream=stream)
            else:
                L.loco_sgd_step(st["cfg"], st["cs"], st["ss"], n, st["p"], 1e-2, stream=stream)

    serial = [make(i, c) for i, c in enumerate(chains)]
    for c, st in zip(chains, serial):
        run(c, st, torch.cuda.current_stream())
    torch.cuda.synchronize()
    together = [make(i, c) for i, c in enumerate(chains)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in chains]
    for c, st, s in zip(chains, together, streams):
        with torch.cuda.stream(s):
            run(c, st, s)
    torch.cuda.synchronize()
    for c, a, b in zip(chains, serial, together):
        for key in ("mean", "p", "m", "v"):
            assert torch.equal(a[key].view(torch.int32), b[key].view(torch.int32)), (c, key)
        for x, y in zip(a["cs"] + a["ss"], b["cs"] + b["ss"]):
            assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), c
