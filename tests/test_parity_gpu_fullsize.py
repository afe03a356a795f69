"""CUDA path vs. CPU oracle on the five workloads at their full sizes, compared
in full.

Each library call runs over the whole bucket in the launch configuration the
benchmark times (the grid depends only on n and the kernel).  The oracle then
recomputes EVERY quant block of every rank and step, chunk by chunk (chunks
are block-aligned, and blocks are independent), from host copies of the
seeded inputs and from its own state: its compensation error of the previous
step and its own codes and steps, which are kept in device memory purely as
storage between steps.  Every output byte -- codes, steps, error, mean,
param/m/v -- must match bit for bit.  Whole-bucket properties that hold at any
size are checked as well (zero experts give zero codes, steps and error).
"""
import gc
import os

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import Stage, assert_bits_equal

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CH = 1 << 27                      # elements per comparison chunk (a multiple of every block size)
THREADS = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import loco
    torch.cuda.set_device(DEV)
    return loco


@pytest.fixture(scope="module")
def stage():
    s = Stage()
    yield s
    s.bufs.clear()


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def W_():
    from bit_gradient_compression_gb300 import workloads
    return workloads


def _gdt(t):
    return np.uint16 if t.dtype == torch.bfloat16 else np.float32


def _chunks(n):
    for e0 in range(0, n, CH):
        yield e0, min(e0 + CH, n)


def check_compress(stage, okw, n, g, err_gpu, codes, scales, step, tag, e_prev=None, oerr=None, ocodes=None,
                   oscales=None):
    """Compare one loco_compress call that has already run with the oracle on
    every block.  The oracle's previous error comes from `oerr` (its own state,
    device storage; updated in place for the next step), else from `e_prev`
    (the seeded input error), else is zero.  The oracle's codes and steps are
    stored into ocodes / oscales when given (inputs of the receiver checks)."""
    bits, block = okw["bits"], okw["block"]
    for e0, e1 in _chunks(n):
        m = e1 - e0
        nbm = -(-m // block)
        c0, cb, s0 = e0 * bits // 8, nbm * block * bits // 8, e0 // block
        g_h = stage.fetch("g", g[e0:e1], _gdt(g))
        if oerr is not None:
            e_h = stage.fetch("e", oerr[e0:e1], np.float32)
        elif e_prev is not None:
            e_h = stage.fetch("e", e_prev[e0:e1], np.float32)
        else:
            e_h = stage.zeros("e", m, np.float32)
        oc = stage.array("oc", cb, np.uint8)
        os_ = stage.array("os", nbm, np.float32)
        oracle.compress(g_h, e_h, step, threads=THREADS, codes=oc, scales=os_, **okw)
        assert_bits_equal(stage.fetch("c", codes[c0:c0 + cb], np.uint8), oc, f"codes {tag} @{e0}")
        assert_bits_equal(stage.fetch("s", scales[s0:s0 + nbm], np.float32), os_, f"scales {tag} @{e0}")
        assert_bits_equal(stage.fetch("ge", err_gpu[e0:e1], np.float32), e_h, f"err {tag} @{e0}")
        if oerr is not None:
            stage.put(oerr[e0:e1], e_h)
        if ocodes is not None:
            stage.put(ocodes[c0:c0 + cb], oc)
            stage.put(oscales[s0:s0 + nbm], os_)


def _rank_rows(stage, codes, scales, e0, e1, bits, block):
    m = e1 - e0
    nbm = -(-m // block)
    c0, cb, s0 = e0 * bits // 8, nbm * block * bits // 8, e0 // block
    rows = [stage.fetch(f"rc{r}", c[c0:c0 + cb], np.uint8) for r, c in enumerate(codes)]
    srows = [stage.fetch(f"rs{r}", s[s0:s0 + nbm], np.float32) for r, s in enumerate(scales)]
    return rows, srows


def check_decode(stage, bits, block, n, mean, ocodes, oscales, tag):
    """Every mean element against the oracle's average of its own codes and steps."""
    for e0, e1 in _chunks(n):
        rows, srows = _rank_rows(stage, ocodes, oscales, e0, e1, bits, block)
        om = oracle.decode_reduce(rows, srows, e1 - e0, bits=bits, block=block, threads=THREADS)
        assert_bits_equal(stage.fetch("mean", mean[e0:e1], np.float32), om, f"mean {tag} @{e0}")


def check_adam(stage, bits, block, n, p, m, v, p0, m0, v0, ocodes, oscales, hpk, t, tag):
    """Every param/m/v element of an Adam step that has run, against the oracle
    started from the state before it (p0, m0, v0; m0/v0 None = zeros)."""
    for e0, e1 in _chunks(n):
        rows, srows = _rank_rows(stage, ocodes, oscales, e0, e1, bits, block)
        ph = stage.fetch("p0", p0[e0:e1], np.float32)
        mh = stage.fetch("m0", m0[e0:e1], np.float32) if m0 is not None else stage.zeros("m0", e1 - e0, np.float32)
        vh = stage.fetch("v0", v0[e0:e1], np.float32) if v0 is not None else stage.zeros("v0", e1 - e0, np.float32)
        oracle.adam_step(rows, srows, e1 - e0, ph, mh, vh, t, bits=bits, block=block, threads=THREADS, **hpk)
        assert_bits_equal(stage.fetch("p", p[e0:e1], np.float32), ph, f"param {tag} @{e0}")
        assert_bits_equal(stage.fetch("m", m[e0:e1], np.float32), mh, f"m {tag} @{e0}")
        assert_bits_equal(stage.fetch("v", v[e0:e1], np.float32), vh, f"v {tag} @{e0}")


ADAM = dict(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, bias_correction=True, eps_inside_sqrt=False)


def test_llama2_7b_fullsize(L, stage):
    """Llama-2-7B-shaped bf16 bucket (6,738,415,616 elements), 4-bit, block 256,
    W = 8 ranks: 8 compress calls, then decode-reduce and the fused Adam step,
    every block compared."""
    w = W_().LLAMA2_7B
    n, bits, block, W = w.n, w.bits, w.block, w.W
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=512)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0, reset_period=512)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    e = torch.empty(n, dtype=torch.float32, device=DEV)
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    scales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    ocodes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    oscales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    for r in range(W):
        w.fill(g, W_().seed_for(7, 1, r))
        e.zero_()
        L.loco_compress(cfg, g, e, 1, codes[r], scales[r])
        check_compress(stage, okw, n, g, e, codes[r], scales[r], 1, f"7b rank {r}", ocodes=ocodes[r],
                       oscales=oscales[r])
    del g, e
    gc.collect()
    torch.cuda.empty_cache()
    mean = torch.empty(n, dtype=torch.float32, device=DEV)
    L.loco_decode_reduce(cfg, codes, scales, n, mean)
    check_decode(stage, bits, block, n, mean, ocodes, oscales, "7b")
    p = W_().fill_uniform(torch.empty(n, device=DEV), 3, -0.02, 0.02)
    m = torch.zeros(n, device=DEV)
    v = torch.zeros(n, device=DEV)
    L.loco_adam_step(cfg, codes, scales, n, p, m, v, L.make_adam(**ADAM), 1)
    p0 = W_().fill_uniform(mean, 3, -0.02, 0.02)          # the parameters before the step, regenerated
    check_adam(stage, bits, block, n, p, m, v, p0, None, None, ocodes, oscales, ADAM, 1, "7b")


def _multi_step(L, stage, w, base_seed, extra_check=None):
    n, bits, block, W = w.n, w.bits, w.block, w.W
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0, reset_period=3)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0, reset_period=3)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    errs = [torch.zeros(n, dtype=torch.float32, device=DEV) for _ in range(W)]
    oerrs = [torch.zeros(n, dtype=torch.float32, device=DEV) for _ in range(W)]   # the oracle's error state
    codes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    scales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    ocodes = [torch.empty(cb, dtype=torch.uint8, device=DEV) for _ in range(W)]
    oscales = [torch.empty(nb, dtype=torch.float32, device=DEV) for _ in range(W)]
    mean = torch.empty(n, dtype=torch.float32, device=DEV)
    for k in range(1, w.steps + 1):
        for r in range(W):
            w.fill(g, W_().seed_for(base_seed, k, r))
            L.loco_compress(cfg, g, errs[r], k, codes[r], scales[r])
            check_compress(stage, okw, n, g, errs[r], codes[r], scales[r], k, f"{w.name} step {k} rank {r}",
                           oerr=oerrs[r], ocodes=ocodes[r], oscales=oscales[r])
            if extra_check:
                extra_check(codes[r], scales[r], errs[r])
        L.loco_decode_reduce(cfg, codes, scales, n, mean)
        check_decode(stage, bits, block, n, mean, ocodes, oscales, f"{w.name} step {k}")


def test_tinyllama_fullsize(L, stage):
    """TinyLlama-1.1B-shaped bf16 bucket, 8-bit, block 128, W = 8, 4 steps
    (reset period 3 so the reset fires at step 3), every block compared."""
    _multi_step(L, stage, W_().TINYLLAMA, 11)


def test_mixtral_moe_fullsize(L, stage):
    """One Mixtral-8x7B MoE layer, Student-t(3) bf16 gradients, experts 3 and 7
    all zero, 4-bit, block 128, W = 8, 4 steps, every block compared."""
    w = W_().MIXTRAL_MOE
    per_expert = 3 * 14336 * 4096
    bits, block = w.bits, w.block

    def zero_experts(codes, scales, err):
        for ex in (3, 7):
            lo, hi = ex * per_expert, (ex + 1) * per_expert
            assert not bool(err[lo:hi].any())
            assert not bool(scales[lo // block:hi // block].any())
            assert not bool(codes[lo * bits // 8:hi * bits // 8].any())

    _multi_step(L, stage, w, 23, extra_check=zero_experts)


@pytest.mark.parametrize("n", [1 << 31, (1 << 31) + 37])
@pytest.mark.parametrize("dtype,bits,block", [(torch.float32, 8, 64), (torch.bfloat16, 4, 256)])
def test_sweep_max_size_compress(L, stage, n, dtype, bits, block):
    """Largest sweep size (2^31 elements; byte offsets need 64-bit indexing), a
    nonzero incoming error, every block compared."""
    cfg = L.make_config(bits=bits, block=block, beta=0.9, err_scale_mult=4.0)
    okw = dict(bits=bits, block=block, beta=0.9, kappa=4.0)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = W_().fill_flat_normal(torch.empty(n, dtype=dtype, device=DEV), 5, outlier_p=1e-3)
    e = W_().fill_flat_normal(torch.empty(n, dtype=torch.float32, device=DEV), 6, sigma=1e-5)
    e_prev = e.clone()
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    scales = torch.empty(nb, dtype=torch.float32, device=DEV)
    L.loco_compress(cfg, g, e, 1, codes, scales)
    check_compress(stage, okw, n, g, e, codes, scales, 1, f"n={n}", e_prev=e_prev)


@pytest.mark.parametrize("W,bits,block", [(16, 4, 256), (1, 8, 64), (8, 4, 128)])
def test_sweep_max_size_decode_and_adam(L, stage, W, bits, block):
    """2^31 + 37 elements of seeded random codes and steps: decode-reduce of W
    ranks and (W <= 8) two fused Adam steps, every element compared."""
    n = (1 << 31) + 37
    cfg = L.make_config(bits=bits, block=block)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(W)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    scales = [torch.rand(nb, device=DEV, generator=gen) * 1e-3 for _ in range(W)]
    mean = torch.empty(n, device=DEV)
    L.loco_decode_reduce(cfg, codes, scales, n, mean)
    check_decode(stage, bits, block, n, mean, codes, scales, f"n={n} W={W}")
    del mean
    if W <= 8:
        p = W_().fill_uniform(torch.empty(n, device=DEV), 1, -0.02, 0.02)
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        p0 = p.clone()
        L.loco_adam_step(cfg, codes, scales, n, p, m, v, L.make_adam(**ADAM), 1)
        check_adam(stage, bits, block, n, p, m, v, p0, None, None, codes, scales, ADAM, 1, f"n={n} W={W}")
        p0.copy_(p)
        m0, v0 = m.clone(), v.clone()
        L.loco_adam_step(cfg, codes, scales, n, p, m, v, L.make_adam(**ADAM), 2)
        check_adam(stage, bits, block, n, p, m, v, p0, m0, v0, codes, scales, ADAM, 2, f"n={n} W={W} t=2")


@pytest.mark.parametrize("log2n", [16, 18, 20, 22, 24])
def test_sweep_sizes_full_compare(L, log2n):
    """Sweep sizes with every combination: bits {4, 8} x block {64, 128, 256} x
    {fp32, bf16} compress and W {1, 2, 4, 8, 16} decode-reduce, compared in full."""
    from tests.helpers import grad_to_np
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


def test_llama2_7b_fullsize_e8(L, stage):
    """The 7B bucket with the 8-bit compensation-error storage, two steps from
    zero state, every block compared (the oracle keeps its own int8 error and
    steps in device storage between the steps)."""
    w = W_().LLAMA2_7B
    n, bits, block = w.n, w.bits, w.block
    cfg = L.make_config(bits=bits, block=block, beta=0.1, err_scale_mult=4.0, reset_period=512)
    okw = dict(bits=bits, block=block, beta=0.1, kappa=4.0, reset_period=512)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    g = torch.empty(n, dtype=w.grad_dtype, device=DEV)
    qe = torch.zeros(n, dtype=torch.int8, device=DEV)
    de = torch.zeros(nb, dtype=torch.float32, device=DEV)
    oqe = torch.zeros(n, dtype=torch.int8, device=DEV)
    ode = torch.zeros(nb, dtype=torch.float32, device=DEV)
    codes = torch.empty(cb, dtype=torch.uint8, device=DEV)
    scales = torch.empty(nb, dtype=torch.float32, device=DEV)
    for k in (1, 2):
        w.fill(g, W_().seed_for(7, k, 0))
        L.loco_compress_e8(cfg, g, qe, de, k, codes, scales)
        for e0, e1 in _chunks(n):
            m = e1 - e0
            nbm = -(-m // block)
            c0, cbm, s0 = e0 * bits // 8, nbm * block * bits // 8, e0 // block
            g_h = stage.fetch("g", g[e0:e1], np.uint16)
            qe_h = stage.fetch("e", oqe[e0:e1], np.int8)
            de_h = stage.fetch("de", ode[s0:s0 + nbm], np.float32)
            oc = stage.array("oc", cbm, np.uint8)
            os_ = stage.array("os", nbm, np.float32)
            oracle.compress_e8(g_h, qe_h, de_h, k, threads=THREADS, codes=oc, scales=os_, **okw)
            tag = f"e8 step {k} @{e0}"
            assert_bits_equal(stage.fetch("c", codes[c0:c0 + cbm], np.uint8), oc, "codes " + tag)
            assert_bits_equal(stage.fetch("s", scales[s0:s0 + nbm], np.float32), os_, "scales " + tag)
            assert_bits_equal(stage.fetch("ge", qe[e0:e1], np.int8), qe_h, "err codes " + tag)
            assert_bits_equal(stage.fetch("gd", de[s0:s0 + nbm], np.float32), de_h, "err steps " + tag)
            stage.put(oqe[e0:e1], qe_h)
            stage.put(ode[s0:s0 + nbm], de_h)


def test_sweep_max_size_sgd_bf16(L, stage):
    """LoCo-SGD with the bf16 parameter copy at 2^31 + 37 elements (W = 4,
    8-bit, block 128), every element compared."""
    n, W, bits, block = (1 << 31) + 37, 4, 8, 128
    cfg = L.make_config(bits=bits, block=block)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(77)
    codes = [torch.randint(0, 256, (cb,), dtype=torch.uint8, device=DEV, generator=gen) for _ in range(W)]
    scales = [torch.rand(nb, device=DEV, generator=gen) * 1e-3 for _ in range(W)]
    p = W_().fill_uniform(torch.empty(n, device=DEV), 2, -0.02, 0.02)
    p0 = p.clone()
    pb = torch.empty(n, dtype=torch.int16, device=DEV)
    L.loco_sgd_step(cfg, codes, scales, n, p, 1e-2, param_bf16=pb)
    for e0, e1 in _chunks(n):
        rows, srows = _rank_rows(stage, codes, scales, e0, e1, bits, block)
        ph = stage.fetch("p0", p0[e0:e1], np.float32)
        pb_h = stage.array("pb0", e1 - e0, np.uint16)
        oracle.sgd_step(rows, srows, e1 - e0, ph, bits=bits, block=block, lr=1e-2, param_bf16=pb_h, threads=THREADS)
        assert_bits_equal(stage.fetch("p", p[e0:e1], np.float32), ph, f"sgd param @{e0}")
        assert_bits_equal(stage.fetch("pb", pb[e0:e1], np.uint16), pb_h, f"sgd bf16 @{e0}")
