"""Pins of the oracle's 8-bit error storage (§3.2 Eqn 7: the compensation
error is kept as compressor(e~; s_e, 8) with s_e = kappa*s, one step per block).

  worked examples ................... tests/golden (cases F, G, H), hand-derived, exact
  agreement with the fp32-error path  when every error lands on the 8-bit grid (kappa = 8
                                      with the dyadic closed-form trace), codes and decoded
                                      errors are identical over 8 steps
  error rounding .................... brute force over all 256 codes (exact rationals)
  zero gradient, reset, resume ...... special cases
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.test_oracle_golden import _bf16_bits, _expected_codes, _grad
from tests.test_oracle_pins import f32_nearest, unpack_codes


def _e8_state(n, block):
    return np.zeros(n, dtype=np.int8), np.zeros(oracle.num_blocks(n, block), dtype=np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_e8_worked_examples(golden, dtype):
    for case in golden["compress_e8_cases"]:
        g = _grad(case)
        gin = g if dtype == "f32" else _bf16_bits(g)
        qe, de = _e8_state(case["n"], case["block"])
        kw = dict(bits=case["bits"], block=case["block"], beta=case["beta"], kappa=case["kappa"],
                  reset_period=case["reset_period"])
        if case["scale_mode"] == "fixed":
            kw["fixed_scale"] = case["fixed_scale"]
        for st in case["steps"]:
            codes, scales = oracle.compress_e8(gin, qe, de, st["step"], **kw)
            exp = _expected_codes(st["codes_head_exact_hex"], case["n"], case["bits"], case["block"])
            assert codes.tobytes() == exp.tobytes(), (case["name"], st["step"])
            assert np.all(scales == np.float32(st["scale_units"] * case["unit"]))
            head = st["err_codes_head"]
            assert list(qe[:len(head)]) == head, (case["name"], st["step"], qe[:8])
            assert not qe[len(head):].any()
            assert np.all(de == np.float32(st["err_step_units"] * case["unit"])), (case["name"], de)


def test_e8_equals_fp32_path_on_the_grid():
    """The closed-form trace's errors are multiples of (1-beta)*x = Delta/8
    (beta = 1/2) or Delta/16 (beta = 3/4); with kappa = 8 resp. 16 they are on
    the 8-bit grid Delta/kappa, so storing them in 8 bits loses nothing: codes and
    decoded errors must equal the fp32-error path step for step."""
    for beta, kappa in ((0.5, 8.0), (0.75, 16.0)):
        block, bits = 64, 4
        delta = 2.0 ** -12
        x = delta / 4
        g = np.zeros(block, dtype=np.float32)
        g[0] = 7 * delta
        g[1:33] = x
        g[33:] = -x
        err = np.zeros(block, dtype=np.float32)
        qe, de = _e8_state(block, block)
        for k in range(1, 9):
            c32, s32 = oracle.compress(g, err, k, bits=bits, block=block, beta=beta, kappa=kappa)
            c8, s8 = oracle.compress_e8(g, qe, de, k, bits=bits, block=block, beta=beta, kappa=kappa)
            assert np.array_equal(c32, c8) and np.array_equal(s32, s8), (beta, k)
            decoded = (qe.astype(np.float32) * de[0]).astype(np.float32)
            assert np.array_equal(decoded, err), (beta, k, decoded[:3], err[:3])


def test_e8_error_rounding_bruteforce():
    """One step from zero state: the fp32 path gives t exactly (err, unclipped);
    the 8-bit path must store the code nearest to t * s_e (halves to even,
    saturated to [-128, 127]) with s_e = kappa * inv_b formed in fp32."""
    rng = np.random.default_rng(21)
    bits, block = 4, 64
    for trial in range(60):
        n = block
        g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, -2)).astype(np.float32)
        kappa = float(rng.choice([4.0, 6.0, 0.05]))  # 0.05: s_e tiny -> exercises ties; large t -> saturation
        beta = float(rng.choice([0.0, 0.5, 0.9]))
        err = np.zeros(n, dtype=np.float32)
        oracle.compress(g, err, 1, bits=bits, block=block, beta=beta, kappa=1e-30)  # bounds +-128*Delta*1e30: unclipped t
        qe, de = _e8_state(n, block)
        codes, scales = oracle.compress_e8(g, qe, de, 1, bits=bits, block=block, beta=beta, kappa=kappa)
        A = Fraction(float(np.max(np.abs(g))))
        if A == 0:
            continue
        inv = f32_nearest(Fraction(7) / A)
        kf = Fraction(float(np.float32(kappa)))  # the library receives kappa as fp32
        inv_e = f32_nearest(kf * Fraction(float(inv)))
        assert de[0] == f32_nearest(Fraction(float(scales[0])) / kf)
        for i in range(n):
            xe = Fraction(float(f32_nearest(Fraction(float(err[i])) * Fraction(float(inv_e)))))
            cands = range(-128, 128)
            dists = [abs(xe - c) for c in cands]
            dmin = min(dists)
            best = [c for c, dd in zip(cands, dists) if dd == dmin]
            want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
            assert qe[i] == want, (trial, i, float(xe), qe[i], want)


def test_e8_zero_reset_resume():
    rng = np.random.default_rng(22)
    n, block, bits = 5 * 128 + 19, 128, 8
    z = np.zeros(n, dtype=np.float32)
    qe, de = _e8_state(n, block)
    for k in range(1, 4):
        c, s = oracle.compress_e8(z, qe, de, k, bits=bits, block=block, beta=0.9, kappa=4.0)
        assert not c.any() and not s.any() and not qe.any() and not de.any()
    gs = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(7)]
    # beta weights the previous error: with 8-bit storage at s_e = 6s the new
    # contribution (1-beta)*r <= (1-beta)*Delta/2 must exceed half a step Delta/12
    # to register at all, so this case uses beta = 0.1.
    kw = dict(bits=bits, block=block, beta=0.1, kappa=6.0, reset_period=3)
    qe, de = _e8_state(n, block)
    full = []
    for k, g in enumerate(gs, start=1):
        full.append(oracle.compress_e8(g, qe, de, k, **kw))
        if k % 3 == 0:
            assert not qe.any()
        else:
            assert qe.any()
    # resume from the state after step 4
    qe2, de2 = _e8_state(n, block)
    for k in range(1, 5):
        oracle.compress_e8(gs[k - 1], qe2, de2, k, **kw)
    for k in range(5, 8):
        c, s = oracle.compress_e8(gs[k - 1], qe2, de2, k, **kw)
        assert np.array_equal(c, full[k - 1][0]) and np.array_equal(s, full[k - 1][1])
    assert np.array_equal(qe2, qe) and np.array_equal(de2, de)


@pytest.mark.parametrize("e8", [False, True])
@pytest.mark.parametrize("bits,block", [(4, 64), (8, 128)])
def test_blocks_are_independent_over_steps(e8, bits, block):
    """Every quant block is its own problem (§3.1: the scale, the codes and the
    error of a block depend on that block's elements only).  A bucket of several
    blocks with very different magnitudes, compressed over 5 steps, gives exactly
    what compressing each block as a bucket of its own gives -- codes, steps and
    the stored error -- including a ragged last block.  Any read of a neighbouring
    block's state (scale, error step, error) breaks it."""
    nblk = 5
    n = nblk * block - 7
    rng = np.random.default_rng(11 + bits + block + int(e8))
    mags = np.float32(10.0) ** np.arange(-4, 1, dtype=np.float32)       # one magnitude per block
    kw = dict(bits=bits, block=block, beta=0.3, kappa=4.0, reset_period=0)
    grads = [(rng.standard_normal(n).astype(np.float32) * np.repeat(mags, block)[:n]) for _ in range(5)]

    def run(lo, hi):
        m = hi - lo
        if e8:
            qe, de = _e8_state(m, block)
        else:
            err = np.zeros(m, dtype=np.float32)
        out = []
        for k, g in enumerate(grads, start=1):
            if e8:
                c, s = oracle.compress_e8(np.ascontiguousarray(g[lo:hi]), qe, de, k, **kw)
                out.append((c.copy(), s.copy(), qe.copy(), de.copy()))
            else:
                c, s = oracle.compress(np.ascontiguousarray(g[lo:hi]), err, k, **kw)
                out.append((c.copy(), s.copy(), err.copy()))
        return out

    whole = run(0, n)
    cb = block * bits // 8
    for b in range(nblk):
        lo, hi = b * block, min(n, (b + 1) * block)
        alone = run(lo, hi)
        for k in range(len(grads)):
            assert whole[k][0][b * cb:(b + 1) * cb].tobytes() == alone[k][0].tobytes(), ("codes", b, k)
            assert whole[k][1][b].view(np.uint32) == alone[k][1][0].view(np.uint32), ("step", b, k)
            if e8:
                assert np.array_equal(whole[k][2][lo:hi], alone[k][2]), ("error codes", b, k)
                assert whole[k][3][b].view(np.uint32) == alone[k][3][0].view(np.uint32), ("error step", b, k)
            else:
                assert np.array_equal(whole[k][2][lo:hi].view(np.uint32), alone[k][2].view(np.uint32)), ("error", b, k)
