"""Exhaustive check of the quotient the receivers use for the rank average's
division by W when W is not a power of two (the division of Eqn 8's fp32 sum
by W, §3.3 of the LoCo paper, which the oracle takes as one IEEE division).

For W in RANK_DIV_FMA the kernels form RN(x / W) as fma(x, zh, RN(x * zl))
with zh the binary32 number just below 1/W and zl = RN(1/W - zh) > 0: the
division by a constant known in advance of Brisebarre, Muller and Raina
("Accelerating correctly rounded floating-point division when the divisor is
known in advance", IEEE Trans. Computers 53(8), 2004), which is correctly
rounded for every x for some divisors and not for others, and which fails near
the bottom of the range where x*zl underflows.  The kernels use it only for
blocks whose steps guarantee |x| >= 2^-100 for every nonzero sum (otherwise
they divide), and zl > 0 keeps the sign of a zero sum.  This test evaluates
the expression for EVERY finite binary32 x with |x| >= 2^-100, and for +-0,
and compares it with the correctly rounded quotient, for every W from 3 to 15
that is not a power of two: each W the kernels admit must give no mismatch.  Reference: x / W in binary64 rounded to binary32 (double
rounding is innocuous for a quotient of two binary32 values, since
53 >= 2*24 + 2).  Candidate: x*zh is exact in binary64 (48 bits), so
x*zh + RN(x*zl) rounded to binary64 and then to binary32 is the fma unless the
binary64 sum lands exactly on a binary32 midpoint; those elements (if any) are
settled in exact rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

RANK_DIV_FMA = (3, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15)   # the rank counts the kernels divide with the fma pair
CANDIDATES = (3, 5, 6, 7, 9, 10, 11, 12, 13, 14, 15)
RANK_DIV_MIN = 2.0 ** -100   # smaller |x| take the IEEE division in the kernels
DEV = torch.device("cuda:0")


def constants(W):
    zh = np.float32(1.0) / np.float32(W)                    # RN(1/W), binary32 division
    if float(zh) > 1.0 / W:
        zh = np.nextafter(zh, np.float32(0))                # the binary32 number just below 1/W
    zl = np.float32(1.0 / W - float(zh))                    # RN(1/W - zh), positive
    return zh, zl


def _exact_fma32(x: float, zh: float, q1: float) -> np.float32:
    s = Fraction(x) * Fraction(zh) + Fraction(q1)
    c = np.float32(float(s))
    best = None
    for y in (c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))):
        d = abs(Fraction(float(y)) - s)
        if best is None or d < best[0] or (d == best[0] and (y.view(np.uint32) & 1) == 0):
            best = (d, y)
    return best[1]


def mismatches(W, chunk=1 << 28):
    """Count of finite binary32 x, |x| >= 2^-100, whose fma pair differs from RN(x / W)."""
    zh, zl = constants(W)
    zh_t = torch.tensor(float(zh), dtype=torch.float32, device=DEV)
    zl_t = torch.tensor(float(zl), dtype=torch.float32, device=DEV)
    bad = 0
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device=DEV)
        bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits).to(torch.int32)
        x = bits.view(torch.float32)
        finite = torch.isfinite(x) & (x.abs() >= RANK_DIV_MIN)
        ref = (x.double() / W).float()
        q1 = x * zl_t                                        # RN(x*zl), one binary32 product
        s64 = x.double() * zh_t.double() + q1.double()      # x*zh exact; one binary64 rounding
        cand = s64.float()
        # a binary64 sum exactly on a binary32 midpoint cannot be rounded from binary64: settle exactly
        up = torch.nextafter(cand, torch.full_like(cand, float("inf")))
        dn = torch.nextafter(cand, torch.full_like(cand, float("-inf")))
        mid = ((s64 == (cand.double() + up.double()) / 2) | (s64 == (cand.double() + dn.double()) / 2)) & finite
        diff = (cand.view(torch.int32) != ref.view(torch.int32)) & finite & ~mid
        bad += int(diff.sum())
        for i in torch.nonzero(mid).flatten().tolist():
            xv, qv = float(x[i]), float(q1[i])
            if _exact_fma32(xv, float(zh), qv).view(np.uint32) != ref[i].cpu().numpy().view(np.uint32):
                bad += 1
    return bad


@pytest.mark.gpu
@pytest.mark.parametrize("W", CANDIDATES)
def test_fma_pair_division_is_exact_where_admitted(W):
    n = mismatches(W)
    if W in RANK_DIV_FMA:
        assert n == 0, f"W = {W}: {n} binary32 inputs round differently"


@pytest.mark.parametrize("W", CANDIDATES)
def test_constants_keep_the_sign_of_zero(W):
    """zh < 1/W < zh + zl with zl > 0: for x = +-0 both x*zh and x*zl are zeros
    of x's sign, and a sum of two zeros of one sign is that zero, so the
    quotient of a zero sum keeps its sign as the IEEE division does."""
    zh, zl = constants(W)
    assert float(zh) < 1.0 / W and zl > 0
    for z in (np.float32(0.0), np.float32(-0.0)):
        assert np.signbit(np.float32(z * zl)) == np.signbit(z) and np.signbit(np.float32(z * zh)) == np.signbit(z)
        assert np.signbit(np.float32(z) / np.float32(W)) == np.signbit(z)


def test_step_threshold_bounds_nonzero_sums():
    """The kernels' guard: with every rank's step 0 or >= 2^-77, every decoded
    term RN(q*Delta) and every rounded partial sum is a multiple of 2^-100, so
    a nonzero sum is at least 2^-100 in magnitude.  Checked on sums of terms
    built from steps at and near the threshold, with cancelling codes."""
    rng = np.random.default_rng(3)
    lo = np.float32(2.0 ** -77)
    for _ in range(20000):
        W = int(rng.integers(2, 17))
        steps = lo * (1 + rng.integers(0, 1 << 12, size=W).astype(np.float32) / np.float32(1 << 12))
        steps[rng.random(W) < 0.2] = 0
        q = rng.integers(-8, 8, size=W).astype(np.float32)
        acc = np.float32(0)
        for w in range(W):
            d = np.float32(q[w] * steps[w])
            acc = d if w == 0 else np.float32(acc + d)
        if acc != 0:
            assert abs(float(acc)) >= 2.0 ** -100
            assert float(acc) / 2.0 ** -100 == int(float(acc) / 2.0 ** -100)
