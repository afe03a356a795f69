"""Paper-literal long runs: fixed scale s (2^19 fine-tuning, 2^17 pre-training),
kappa = s_e/s in {4, 6}, reset period T_c in {512, 1024} ("LoCo: Low-Bit
Communication Adaptor for Large-scale Model Training", §3.1 and §3.2 Eqn 7),
over more than 1024 steps so that the reset fires.

CPU (oracle): the stored error stays inside the 8-bit compressor's range at every
step and is exactly zero after every reset step.  GPU: the CUDA path matches
the oracle bit for bit at every step, for both error storages.
"""
import numpy as np
import pytest
import torch

import oracle

STEPS = 1100


def _grads(n, seed):
    rng = np.random.default_rng(seed)
    for k in range(STEPS):
        # heavy-tailed, magnitudes around the fixed scales' ranges
        z = rng.standard_t(3, size=n) * 10.0 ** rng.uniform(-7, -5)
        yield k + 1, z.astype(np.float32)


@pytest.mark.parametrize("s,kappa,Tc", [(2.0 ** 19, 4.0, 512), (2.0 ** 17, 6.0, 1024)])
def test_fixed_scale_long_trace_invariants(s, kappa, Tc):
    n, bits, block = 3000, 4, 128
    err = np.zeros(n, dtype=np.float32)
    delta = np.float32(1.0) / np.float32(s)
    de = np.float32(delta / np.float32(kappa))
    lo, hi = np.float32(-128 * de), np.float32(127 * de)
    for k, g in _grads(n, 5):
        codes, scales = oracle.compress(g, err, k, bits=bits, block=block, beta=0.9, kappa=kappa,
                                        reset_period=Tc, fixed_scale=s)
        assert np.all(scales == delta)
        assert np.all(err >= lo) and np.all(err <= hi)
        if k % Tc == 0:
            assert not err.any(), k


@pytest.mark.gpu
@pytest.mark.parametrize("storage", ["fp32", "int8"])
@pytest.mark.parametrize("s,kappa,Tc,bits", [(2.0 ** 19, 4.0, 512, 4), (2.0 ** 17, 6.0, 1024, 8)])
def test_fixed_scale_long_trace_gpu(storage, s, kappa, Tc, bits):
    from bit_gradient_compression_gb300 import loco as L
    dev = torch.device("cuda:0")
    n, block = 20_003, 128
    beta = 0.9 if storage == "fp32" else 0.3
    cfg = L.make_config(bits=bits, block=block, beta=beta, err_scale_mult=kappa, reset_period=Tc, fixed_scale=s)
    nb, cb = L.loco_num_blocks(n, block), L.loco_code_bytes(n, bits, block)
    codes = torch.empty(cb, dtype=torch.uint8, device=dev)
    scales = torch.empty(nb, device=dev)
    okw = dict(bits=bits, block=block, beta=beta, kappa=kappa, reset_period=Tc, fixed_scale=s)
    if storage == "fp32":
        e = torch.zeros(n, device=dev)
        e_h = np.zeros(n, np.float32)
    else:
        qe, de = torch.zeros(n, dtype=torch.int8, device=dev), torch.zeros(nb, device=dev)
        qe_h, de_h = np.zeros(n, np.int8), np.zeros(nb, np.float32)
    for k, g_h in _grads(n, 9):
        g = torch.from_numpy(g_h).to(dev)
        if storage == "fp32":
            L.loco_compress(cfg, g, e, k, codes, scales)
            oc, os_ = oracle.compress(g_h, e_h, k, **okw)
        else:
            L.loco_compress_e8(cfg, g, qe, de, k, codes, scales)
            oc, os_ = oracle.compress_e8(g_h, qe_h, de_h, k, **okw)
        if k % 50 == 0 or k % Tc in (0, 1) or k > STEPS - 3:
            torch.cuda.synchronize()
            assert np.array_equal(codes.cpu().numpy(), oc), k
            assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32)), k
            if storage == "fp32":
                assert np.array_equal(e.cpu().numpy().view(np.uint32), e_h.view(np.uint32)), k
            else:
                assert np.array_equal(qe.cpu().numpy(), qe_h), k
                assert np.array_equal(de.cpu().numpy().view(np.uint32), de_h.view(np.uint32)), k
