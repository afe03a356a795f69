"""CUDA path vs. CPU oracle on the five workloads at their full sizes.

Each call runs over the whole bucket in the same launch configuration the
benchmark times (the grid depends only on n and the kernel); the oracle then
recomputes a sample of quant blocks -- the first, the last and ~40 random
ones per rank and step -- from host copies of exactly the bytes the kernel
read, and every sampled output must match bit for bit.  Whole-bucket
properties are checked where they hold at any size (zero experts give zero
codes, scales and error everywhere).
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_bits_equal, block_index, code_rows, grad_to_np, sample_block_ids, scale_rows, take

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SAMPLES = 40


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import loco
    torch.cuda.set_device(DEV)
    return loco


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def W_():
    from bit_gradient_compression_gb300 import workloads
    return workloads


class Sampler:
    """Sampled blocks of one bucket and the host copies taken before a call."""

    def __init__(self, n, block, seed):
        self.n, self.block = n, block
        self.nb = -(-n // block)
        self.ids = sample_block_ids(self.nb, SAMPLES, seed)
        self.idx = block_index(self.ids, block, n, DEV)

    def grab(self, t):
        return take(t, self.idx)


def _check_compress(L, cfg, okw, s: Sampler, g, e, step, codes, scales, tag):
    g_h = grad_to_np(s.grab(g))
    e_h = s.grab(e).numpy().copy()
    L.loco_compress(cfg, g, e, step, codes, scales)
    oc, os_ = oracle.compress(g_h, e_h, step, **okw)
    torch.cuda.synchronize()
    assert_bits_equal(code_rows(codes, s.ids, okw["block"], okw["bits"]), oc, "codes " + tag)
    assert_bits_equal(scale_rows(scales, s.ids), os_, "scales " + tag)
    assert_bits_equal(s.grab(e).numpy(), e_h, "err " + tag)
    return oc, os_


def _check_decode(L, cfg, bits, block, s: Sampler, codes, scales, mean, tag):
    L.loco_decode_reduce(cfg, codes, scales, s.n, mean)
    rows = [code_rows(c, s.ids, block, bits) for c in codes]
    srows = [scale_rows(x, s.ids) for x in scales]
    om = oracle.decode_reduce(rows, srows, s.idx.numel(), bits=bits, block=block)
    torch.cuda.synchronize()
    assert_bits_equal(s.grab(mean).numpy(), om, "mean " + tag)


def _check_adam(L, cfg, bits, block, s: Sampler, codes, scales, p, m, v, hpk, t, tag):
    ph, mh, vh = s.grab(p).numpy().copy(), s.grab(m).numpy().copy(), s.grab(v).numpy().copy()
    L.loco_adam_step(cfg, codes, scales, s.n, p, m, v, L.make_adam(**hpk), t)
    rows = [code_rows(c, s.ids, block, bits) for c in codes]
    srows = [scale_rows(x, s.ids) for x in scales]
    oracle.adam_step(rows, srows, s.idx.numel(), ph, mh, vh, t, bits=bits, block=block, **hpk)
    torch.cuda.synchronize()
    assert_bits_equal(s.grab(p).numpy(), ph, "param " + tag)
    assert_bits_equal(s.grab(m).numpy(), mh, "m " + tag)
    assert_bits_equal(s.grab(v).numpy(), vh, "v " + tag)


ADAM = dict(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, bias_correction=True, eps_inside_sqrt=False)


def test_llama2_7b_fullsize(L):
    """Llama-2-7B-shaped bf16 bucket (6,738,415,616 elements), 4-bit, block 256,
    W = 8 ranks: 8 compress calls, then decode-reduce and the fused Adam step."""
    w = W_().LLAMA2_7B
    n, bits, block, W = w.n, w.bits, w.block, w.W
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=512)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0, reset_period=512)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    e = torch.empty(n, dtype=torch.float32, device=DEV)
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    scales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    for r in range(W):
        s = Sampler(n, block, 100 + r)
        w.fill(g, W_().seed_for(7, 1, r))
        e.zero_()
        _check_compress(L, cfg, okw, s, g, e, 1, codes[r], scales[r], f"7b rank {r}")
    del g, e
    s = Sampler(n, block, 999)
    mean = torch.empty(n, dtype=torch.float32, device=DEV)
    _check_decode(L, cfg, bits, block, s, codes, scales, mean, "7b")
    del mean
    p = W_().fill_uniform(torch.empty(n, device=DEV), 3, -0.02, 0.02)
    m = torch.zeros(n, device=DEV)
    v = torch.zeros(n, device=DEV)
    _check_adam(L, cfg, bits, block, s, codes, scales, p, m, v, ADAM, 1, "7b")


def _multi_step(L, w, base_seed, extra_check=None):
    n, bits, block, W = w.n, w.bits, w.block, w.W
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=3)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0, reset_period=3)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    errs = [torch.zeros(n, dtype=torch.float32, device=DEV) for _ in range(W)]
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    scales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    mean = torch.empty(n, dtype=torch.float32, device=DEV)
    for k in range(1, w.steps + 1):
        for r in range(W):
            s = Sampler(n, block, 31 * k + r)
            w.fill(g, W_().seed_for(base_seed, k, r))
            _check_compress(L, cfg, okw, s, g, errs[r], k, codes[r], scales[r], f"{w.name} step {k} rank {r}")
            if extra_check:
                extra_check(codes[r], scales[r], errs[r])
        _check_decode(L, cfg, bits, block, Sampler(n, block, 77 + k), codes, scales, mean, f"{w.name} step {k}")


def test_tinyllama_fullsize(L):
    """TinyLlama-1.1B-shaped bf16 bucket, 8-bit, block 128, W = 8, 4 steps
    (reset period 3 so the reset fires at step 3)."""
    _multi_step(L, W_().TINYLLAMA, 11)


def test_mixtral_moe_fullsize(L):
    """One Mixtral-8x7B MoE layer, Student-t(3) bf16 gradients, experts 3 and 7
    all zero, 4-bit, block 128, W = 8, 4 steps."""
    w = W_().MIXTRAL_MOE
    per_expert = 3 * 14336 * 4096
    bits, block = w.bits, w.block

    def zero_experts(codes, scales, err):
        for ex in (3, 7):
            lo, hi = ex * per_expert, (ex + 1) * per_expert
            assert not bool(err[lo:hi].any())
            assert not bool(scales[lo // block:hi // block].any())
            assert not bool(codes[lo * bits // 8:hi * bits // 8].any())

    _multi_step(L, w, 23, extra_check=zero_experts)


@pytest.mark.parametrize("n", [1 << 31, (1 << 31) + 37])
@pytest.mark.parametrize("dtype,bits,block", [(torch.float32, 8, 64), (torch.bfloat16, 4, 256)])
def test_sweep_max_size_compress(L, n, dtype, bits, block):
    """Largest sweep size (2^31 elements; byte offsets need 64-bit indexing)."""
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = W_().fill_flat_normal(torch.empty(n, dtype=dtype, device=DEV), 5, outlier_p=1e-3)
    e = W_().fill_flat_normal(torch.empty(n, dtype=torch.float32, device=DEV), 6, sigma=1e-5)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    scales = torch.empty(nb, dtype=torch.float32, device=DEV)
    s = Sampler(n, block, 5)
    _check_compress(L, cfg, okw, s, g, e, 1, codes, scales, f"n={n}")


@pytest.mark.parametrize("W,bits,block", [(16, 4, 256), (1, 8, 64), (8, 4, 128)])
def test_sweep_max_size_decode_and_adam(L, W, bits, block):
    n = (1 << 31) + 37
    cfg = L.make_config(bits=bits, block=block)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(W)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    scales = [torch.rand(nb, device=DEV, generator=gen) * 1e-3 for _ in range(W)]
    s = Sampler(n, block, 8)
    mean = torch.empty(n, device=DEV)
    _check_decode(L, cfg, bits, block, s, codes, scales, mean, f"n={n} W={W}")
    del mean
    if W <= 8:
        p = W_().fill_uniform(torch.empty(n, device=DEV), 1, -0.02, 0.02)
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        _check_adam(L, cfg, bits, block, s, codes, scales, p, m, v, ADAM, 1, f"n={n} W={W}")
        _check_adam(L, cfg, bits, block, s, codes, scales, p, m, v, ADAM, 2, f"n={n} W={W} t=2")


@pytest.mark.parametrize("log2n", [16, 18, 20, 22, 24])
def test_sweep_sizes_full_compare(L, log2n):
    """Sweep sizes small enough for the oracle to recompute everything:
    bits {4, 8} x block {64, 128, 256} x {fp32, bf16} compress and
    W {1, 2, 4, 8, 16} decode-reduce, compared in full."""
    n = 1 << log2n
    for dtype in (torch.float32, torch.bfloat16):
        g = W_().fill_flat_normal(torch.empty(n, dtype=dtype, device=DEV), log2n, outlier_p=1e-3)
        g_h = grad_to_np(g)
        for bits in (4, 8):
            for block in (64, 128, 256):
                cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0)
                nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
                e = torch.zeros(n, device=DEV)
                codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
                scales = torch.empty(nb, device=DEV)
                L.loco_compress(cfg, g, e, 1, codes, scales)
                e_h = np.zeros(n, np.float32)
                oc, os_ = oracle.compress(g_h, e_h, 1, bits=bits, block=block, beta=0.9, kappa=4.0, threads=8)
                torch.cuda.synchronize()
                tag = f"n=2^{log2n} {dtype} bits={bits} block={block}"
                assert_bits_equal(codes.cpu().numpy(), oc, "codes " + tag)
                assert_bits_equal(scales.cpu().numpy(), os_, "scales " + tag)
                assert_bits_equal(e.cpu().numpy(), e_h, "err " + tag)
                if dtype == torch.bfloat16:
                    for W in (1, 2, 4, 8, 16):
                        mean = torch.empty(n, device=DEV)
                        L.loco_decode_reduce(cfg, [codes] * W, [scales] * W, n, mean)
                        om = oracle.decode_reduce([oc] * W, [os_] * W, n, bits=bits, block=block, threads=8)
                        torch.cuda.synchronize()
                        assert_bits_equal(mean.cpu().numpy(), om, f"mean W={W} " + tag)


def test_llama2_7b_fullsize_e8(L):
    """The 7B bucket with the 8-bit compensation-error storage, two steps from zero state."""
    w = W_().LLAMA2_7B
    n, bits, block = w.n, w.bits, w.block
    cfg = L.make_config(bits=bits, block=block, beta=0.1, err_scale_mult=4.0, reset_period=512)
    okw = dict(bits=bits, block=block, beta=0.1, kappa=4.0, reset_period=512)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    qe = torch.zeros(n, dtype=torch.int8, device=DEV)
    de = torch.zeros(nb, dtype=torch.float32, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    scales = torch.empty(nb, dtype=torch.float32, device=DEV)
    for k in (1, 2):
        s = Sampler(n, block, 300 + k)
        w.fill(g, W_().seed_for(7, k, 0))
        g_h = grad_to_np(s.grab(g))
        qe_h = s.grab(qe).numpy().copy()
        de_h = scale_rows(de, s.ids).copy()
        L.loco_compress_e8(cfg, g, qe, de, k, codes, scales)
        oc, os_ = oracle.compress_e8(g_h, qe_h, de_h, k, **okw)
        torch.cuda.synchronize()
        assert_bits_equal(code_rows(codes, s.ids, block, bits), oc, f"e8 codes step {k}")
        assert_bits_equal(scale_rows(scales, s.ids), os_, f"e8 scales step {k}")
        assert_bits_equal(s.grab(qe).numpy(), qe_h, f"e8 err codes step {k}")
        assert_bits_equal(scale_rows(de, s.ids), de_h, f"e8 err steps step {k}")


def test_sweep_max_size_sgd_bf16(L):
    """LoCo-SGD with the bf16 parameter copy at 2^31 + 37 elements (W = 4, 8-bit, block 128)."""
    n, W, bits, block = (1 << 31) + 37, 4, 8, 128
    cfg = L.make_config(bits=bits, block=block)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(77)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    scales = [torch.rand(nb, device=DEV, generator=gen) * 1e-3 for _ in range(W)]
    p = W_().fill_uniform(torch.empty(n, device=DEV), 2, -0.02, 0.02)
    pb = torch.empty(n, dtype=torch.int16, device=DEV)
    s = Sampler(n, block, 12)
    ph = s.grab(p).numpy().copy()
    L.loco_sgd_step(cfg, codes, scales, n, p, 1e-2, param_bf16=pb)
    rows = [code_rows(c, s.ids, block, bits) for c in codes]
    srows = [scale_rows(x, s.ids) for x in scales]
    pb_h = np.zeros(s.idx.numel(), dtype=np.uint16)
    oracle.sgd_step(rows, srows, s.idx.numel(), ph, bits=bits, block=block, lr=1e-2, param_bf16=pb_h)
    torch.cuda.synchronize()
    assert_bits_equal(s.grab(p).numpy(), ph, "sgd param")
    assert_bits_equal(s.grab(pb).numpy().view(np.uint16), pb_h, "sgd bf16")
