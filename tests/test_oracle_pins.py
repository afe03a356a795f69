"""Pins of the CPU oracle to facts other than itself.

Method: "LoCo: Low-Bit Communication Adaptor for Large-scale Model Training"
(arXiv 2407.04480).  Which pin covers which step:

  Eqn (1),(3) rounding/saturation/packing .. brute force over all codes (test_bruteforce_*)
  scale Delta = A/qmax, inv = qmax/A ....... exact-rational nearest-fp32 check (test_bruteforce_*)
  Eqn (4) error r = h - d .................. exact reconstruction d + r == h (test_reconstruction_exact)
  Eqn (2) compensation ..................... closed-form traces over steps (test_closed_form_trace_*)
  Eqn (5) moving average ................... closed-form traces; beta=0 telescoping; beta=1 no feedback;
                                             the telescoping identity sum(d-g) = -e_K/(1-beta) (Eqn 6)
  Eqn (7) clip / reset ..................... fixed-scale saturation; reset period; resume
  Eqn (8) average .......................... fp64 shadow bound; W=1; identical ranks; rank permutation
  Eqn (9) Adam ............................. torch.optim.AdamW cross-check; first-step closed form
Worked examples with exact values live in tests/golden (test_oracle_golden.py).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

QMAX = {4: 7, 8: 127}


# ---------------------------------------------------------------- helpers (test-side, independent)

def unpack_codes(codes: np.ndarray, bits: int, n_total: int) -> np.ndarray:
    """Sign-extended integer codes from the packed bytes (low nibble = even element)."""
    if bits == 8:
        return codes.view(np.int8).astype(np.int64)[:n_total]
    lo = (codes & 0xF).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    q = np.empty(codes.size * 2, dtype=np.int64)
    q[0::2] = lo
    q[1::2] = hi
    q = np.where(q >= 8, q - 16, q)
    return q[:n_total]


def f32_nearest(fr: Fraction) -> np.float32:
    """Nearest fp32 to an exact rational, halves to even (exhaustive over neighbours)."""
    c = np.float32(float(fr))
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    best = None
    for x in cands:
        d = abs(Fraction(float(x)) - fr)
        if best is None or d < best[0] or (d == best[0] and (x.view(np.uint32) & 1) == 0):
            best = (d, x)
    return best[1]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the bit patterns."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def run(g, err, step, **kw):
    return oracle.compress(g, err, step, **kw)


# ---------------------------------------------------------------- Eqn (1),(3): brute force

@pytest.mark.parametrize("bits", [4, 8])
def test_bruteforce_tiny(bits):
    rng = np.random.default_rng(1234 + bits)
    qmax, qmin = QMAX[bits], -QMAX[bits] - 1
    block = 64
    for trial in range(300):
        n = int(rng.integers(1, 17))
        if trial % 3 == 0:
            # exact ties: A = qmax * 2^j, elements k/2 * 2^j
            j = int(rng.integers(-20, 0))
            h = (rng.integers(-2 * qmax, 2 * qmax + 1, size=n) / 2.0 * 2.0 ** j).astype(np.float32)
            h[int(rng.integers(0, n))] = np.float32(qmax * 2.0 ** j) * (1 if rng.random() < 0.5 else -1)
        else:
            h = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 1)).astype(np.float32)
        err = np.zeros(n, dtype=np.float32)
        codes, scales = run(h, err, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
        A = Fraction(float(np.max(np.abs(h))))
        if A == 0:
            assert scales[0] == 0 and not codes.any()
            continue
        delta = f32_nearest(A / qmax)
        inv = f32_nearest(Fraction(qmax) / A)
        assert scales[0] == delta, (trial, scales[0], delta)
        q = unpack_codes(codes, bits, block)
        assert np.all(q[n:] == 0), "padding codes must be 0"
        for i in range(n):
            x = f32_nearest(Fraction(float(h[i])) * Fraction(float(inv)))
            xf = Fraction(float(x))
            cands = range(qmin, qmax + 1)
            dists = [abs(xf - c) for c in cands]
            dmin = min(dists)
            best = [c for c, d in zip(cands, dists) if d == dmin]
            want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
            assert q[i] == want, (trial, i, float(h[i]), float(x), q[i], want)
        # the element of largest magnitude lands on +-qmax (absmax scaling)
        imax = int(np.argmax(np.abs(h)))
        assert abs(q[imax]) == qmax


# ---------------------------------------------------------------- Eqn (4): exact reconstruction

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("block", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reconstruction_exact(bits, block, dtype):
    """With beta = 0 the stored error is r = h - d itself (no clip in absmax mode),
    and d + r must give back h exactly, bit for bit."""
    rng = np.random.default_rng(7 + bits + block)
    n = 5 * block + 37  # several blocks and a ragged tail
    err = np.zeros(n, dtype=np.float32)
    for step in range(1, 4):
        g32 = (rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2, size=n)).astype(np.float32)
        g32[rng.random(n) < 0.01] *= 100
        if dtype == "bf16":
            gb = bf16_bits(g32)
            gin, gval = gb, bf16_to_f32(gb)
        else:
            gin, gval = g32, g32
        h = (gval + err).astype(np.float32)  # fp32 sum, as the compensation step states
        codes, scales = run(gin, err, step, bits=bits, block=block, beta=0.0, kappa=4.0)
        q = unpack_codes(codes, bits, n)
        d = (q.astype(np.float32) * np.repeat(scales, block)[:n]).astype(np.float32)
        back = (d + err).astype(np.float32)
        assert np.array_equal(back.view(np.uint32), h.view(np.uint32)) or np.array_equal(back, h)
        assert np.all(np.abs(err) <= np.repeat(scales, block)[:n] * (0.5 + 2.0 ** -20))


# ---------------------------------------------------------------- special inputs

def test_zero_gradient_zero_everything():
    for bits, block in [(4, 256), (8, 128), (4, 64)]:
        n = 3 * block + 5
        g = np.zeros(n, dtype=np.float32)
        err = np.zeros(n, dtype=np.float32)
        for step in range(1, 5):
            codes, scales = run(g, err, step, bits=bits, block=block, beta=0.9, kappa=4.0)
            assert not codes.any() and not scales.any() and not err.any()
            assert not np.signbit(err).any()


def test_zero_blocks_among_nonzero():
    block, bits = 128, 4
    n = 8 * block
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[2 * block:4 * block] = 0
    g[7 * block:] = 0
    err = np.zeros(n, dtype=np.float32)
    for step in range(1, 4):
        codes, scales = run(g, err, step, bits=bits, block=block, beta=0.9, kappa=4.0)
        for b in (2, 3, 7):
            assert scales[b] == 0
            assert not codes[b * 64:(b + 1) * 64].any()
            assert not err[b * block:(b + 1) * block].any()


@pytest.mark.parametrize("bits", [4, 8])
def test_constant_block(bits):
    qmax = QMAX[bits]
    block = 64
    for j in range(-24, 4, 3):
        for sign in (1, -1):
            c = np.float32(sign * qmax * 2.0 ** j)
            g = np.full(block, c, dtype=np.float32)
            err = np.zeros(block, dtype=np.float32)
            codes, scales = run(g, err, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
            q = unpack_codes(codes, bits, block)
            assert np.all(q == sign * qmax)
            assert scales[0] == np.float32(2.0 ** j)
            assert not err.any()  # exact round trip
    rng = np.random.default_rng(11)
    for _ in range(200):
        c = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-8, 2))
        g = np.full(block, c, dtype=np.float32)
        err = np.zeros(block, dtype=np.float32)
        codes, scales = run(g, err, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
        q = unpack_codes(codes, bits, block)
        assert np.all(q == np.sign(c) * qmax)
        d = np.float32(np.float32(q[0]) * scales[0])
        assert abs(float(d) - float(c)) <= float(np.spacing(np.abs(c)))
        assert np.float32(d + err[0]) == c


# ---------------------------------------------------------------- Eqn (2),(5): closed-form traces

# A block holding one element A = qmax * Delta (Delta a power of two) and small elements
# +-x with x = Delta/4, the gradient repeated every step.  A is encoded exactly (r = 0), so
# Delta stays fixed; the small elements follow, by hand:
#   h_k = x + e_{k-1};  q_k = round(h_k / Delta);  r_k = h_k - q_k Delta;
#   e_k = beta e_{k-1} + (1-beta) r_k.
# beta = 1/2:  e/x = 0.5, 1, 1.5, 0, 0.5, 1, 1.5, 0      q = 0,0,0,1,0,0,0,1
#   (k=3: h = 2x = Delta/2 is a tie and rounds to 0; k=4: h = 2.5x -> q = 1, r = -1.5x, e = 0)
# beta = 3/4:  e/x = .25, .5, .75, 1, 1.25, .5, .75, 1   q = 0,0,0,0,0,1,0,0
#   (k=5: h = 2x tie -> 0; k=6: h = 2.25x -> q = 1, r = -1.75x, e = .9375x - .4375x = .5x)
TRACES = {
    0.5: ([0.5, 1, 1.5, 0, 0.5, 1, 1.5, 0], [0, 0, 0, 1, 0, 0, 0, 1]),
    0.75: ([0.25, 0.5, 0.75, 1, 1.25, 0.5, 0.75, 1], [0, 0, 0, 0, 0, 1, 0, 0]),
}


@pytest.mark.parametrize("beta", [0.5, 0.75])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_closed_form_trace_dyadic(beta, bits, dtype):
    qmax = QMAX[bits]
    block = 64
    delta = 2.0 ** -12
    x = delta / 4
    g = np.zeros(block, dtype=np.float32)
    g[0] = qmax * delta
    g[1:33] = x
    g[33:] = -x
    gin = g if dtype == "f32" else bf16_bits(g)
    err = np.zeros(block, dtype=np.float32)
    e_units, q_small = TRACES[beta]
    for k in range(1, 9):
        codes, scales = run(gin, err, k, bits=bits, block=block, beta=beta, kappa=4.0)
        q = unpack_codes(codes, bits, block)
        assert scales[0] == np.float32(delta)
        assert q[0] == qmax and err[0] == 0
        assert np.all(q[1:33] == q_small[k - 1]) and np.all(q[33:] == -q_small[k - 1]), (k, q[:3])
        assert np.all(err[1:33] == np.float32(e_units[k - 1] * x)), (k, err[1] / x)
        assert np.all(err[33:] == np.float32(-e_units[k - 1] * x)), k


def test_closed_form_trace_beta09():
    """beta = 0.9: while q stays 0 the error grows by (1-beta) x per step, e_k = 0.1 k x."""
    block, bits = 64, 4
    delta = 2.0 ** -12
    x = delta / 4
    g = np.zeros(block, dtype=np.float32)
    g[0] = 7 * delta
    g[1:] = x
    err = np.zeros(block, dtype=np.float32)
    for k in range(1, 11):  # h_k = x (1 + 0.1 (k-1)) <= 1.9 x < Delta/2
        codes, _ = run(g, err, k, bits=bits, block=block, beta=0.9, kappa=4.0)
        assert np.all(unpack_codes(codes, bits, block)[1:] == 0)
        np.testing.assert_allclose(err[1:], 0.1 * k * x, rtol=1e-6)


# ---------------------------------------------------------------- special cases of beta

def _random_grads(rng, n, steps, scale=1e-3):
    return [(rng.standard_normal(n) * scale).astype(np.float32) for _ in range(steps)]


def test_beta0_is_plain_error_feedback_telescoping():
    """beta = 0 is Seide et al.'s EFC (Eqn 4): sum_k d_k + e_K = sum_k g_k up to the
    rounding of the compensation sums."""
    rng = np.random.default_rng(5)
    n, block, bits, K = 4 * 256 + 3, 256, 4, 20
    err = np.zeros(n, dtype=np.float32)
    sd = np.zeros(n)
    sg = np.zeros(n)
    hmax = 0.0
    for k, g in enumerate(_random_grads(rng, n, K), start=1):
        hmax = max(hmax, float(np.max(np.abs(g + err))))
        codes, scales = run(g, err, k, bits=bits, block=block, beta=0.0, kappa=4.0)
        q = unpack_codes(codes, bits, n)
        sd += (q.astype(np.float32) * np.repeat(scales, block)[:n]).astype(np.float32)
        sg += g
    assert np.max(np.abs(sd + err - sg)) <= K * hmax * 2.0 ** -23


def test_beta1_means_no_feedback():
    """beta = 1 keeps e = 0: every step compresses g alone (no error feedback)."""
    rng = np.random.default_rng(6)
    n, block, bits = 3 * 128 + 9, 128, 4
    err = np.zeros(n, dtype=np.float32)
    for k, g in enumerate(_random_grads(rng, n, 5), start=1):
        codes, scales = run(g, err, k, bits=bits, block=block, beta=1.0, kappa=4.0)
        assert not err.any()
        c0, s0 = run(g, np.zeros(n, dtype=np.float32), 1, bits=bits, block=block, beta=0.0, kappa=4.0)
        assert np.array_equal(codes, c0) and np.array_equal(scales, s0)


def test_non_accumulation_identity_eqn6():
    """With beta < 1 and no clipping, d_k = h_k - r_k and e_k = beta e_{k-1} + (1-beta) r_k give
    sum_k (d_k - g_k) = (e_0 - e_K)/(1-beta): the accumulated compression error stays of the
    size of one error (Eqn 6).  Without feedback (beta = 1) it is a random walk."""
    rng = np.random.default_rng(8)
    n, block, bits, K = 2048, 256, 4, 200
    for beta in (0.0, 0.5, 0.9):
        err = np.zeros(n, dtype=np.float32)
        acc = np.zeros(n)
        hsum = 0.0
        for k, g in enumerate(_random_grads(rng, n, K), start=1):
            hsum += float(np.max(np.abs(g + err)))
            codes, scales = run(g, err, k, bits=bits, block=block, beta=beta, kappa=4.0)
            q = unpack_codes(codes, bits, n)
            acc += (q.astype(np.float32) * np.repeat(scales, block)).astype(np.float64) - g
        resid = acc + err.astype(np.float64) / (1.0 - beta)
        assert np.max(np.abs(resid)) <= 4 * hsum * 2.0 ** -24 / (1.0 - beta), beta
        bounded = np.linalg.norm(acc)
    err = np.zeros(n, dtype=np.float32)
    acc = np.zeros(n)
    for k, g in enumerate(_random_grads(rng, n, K), start=1):
        codes, scales = run(g, err, k, bits=bits, block=block, beta=1.0, kappa=4.0)
        q = unpack_codes(codes, bits, n)
        acc += (q.astype(np.float32) * np.repeat(scales, block)).astype(np.float64) - g
    assert np.linalg.norm(acc) > 3 * bounded


# ---------------------------------------------------------------- Eqn (7): clip and reset

def test_fixed_scale_saturation_hits_bounds():
    s, kappa, block, bits = 2.0 ** 19, 4.0, 64, 4
    rng = np.random.default_rng(9)
    n = 10 * block
    g = (rng.standard_normal(n) * 1e-4).astype(np.float32)  # |h| >> 7/s: most codes saturate
    err = np.zeros(n, dtype=np.float32)
    codes, scales = run(g, err, 1, bits=bits, block=block, beta=0.0, kappa=kappa, fixed_scale=s)
    de = np.float32(np.float32(1.0 / s) / np.float32(kappa))
    lo, hi = np.float32(-128 * de), np.float32(127 * de)
    assert np.all(scales == np.float32(1.0 / s))
    assert np.all(err >= lo) and np.all(err <= hi)
    assert np.any(err == lo) and np.any(err == hi)
    q = unpack_codes(codes, bits, n)
    big = np.abs(g) * s > 8
    assert np.all(q[big] == np.where(g[big] > 0, 7, -8))


def test_reset_period():
    rng = np.random.default_rng(10)
    n, block, bits, Tc = 2 * 256 + 17, 256, 4, 3
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    err = np.zeros(n, dtype=np.float32)
    hist = []
    for k in range(1, 8):
        codes, scales = run(g, err, k, bits=bits, block=block, beta=0.9, kappa=4.0, reset_period=Tc)
        hist.append((codes.copy(), scales.copy(), err.copy()))
        if k % Tc == 0:
            assert not err.any()
        else:
            assert err.any()
    # after a reset, the next step repeats step 1
    for k_after in (4, 7):
        assert np.array_equal(hist[k_after - 1][0], hist[0][0])
        assert np.array_equal(hist[k_after - 1][2], hist[0][2])


def test_resume_from_checkpoint():
    """The error buffer and the step counter are the whole sender state."""
    rng = np.random.default_rng(12)
    n, block, bits = 3 * 128 + 1, 128, 8
    gs = _random_grads(rng, n, 6)
    kw = dict(bits=bits, block=block, beta=0.9, kappa=6.0, reset_period=4)
    err = np.zeros(n, dtype=np.float32)
    full = [run(g, err, k, **kw) for k, g in enumerate(gs, start=1)]
    e_full = err.copy()
    err2 = np.zeros(n, dtype=np.float32)
    for k in range(1, 4):
        run(gs[k - 1], err2, k, **kw)
    ckpt = err2.copy()
    err3 = ckpt.copy()
    for k in range(4, 7):
        c, s = run(gs[k - 1], err3, k, **kw)
        assert np.array_equal(c, full[k - 1][0]) and np.array_equal(s, full[k - 1][1])
    assert np.array_equal(err3, e_full)


# ---------------------------------------------------------------- Eqn (8): average of W ranks

def _ranks(rng, n, W, bits, block):
    codes, scales = [], []
    for w in range(W):
        g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2)).astype(np.float32)
        c, s = run(g, np.zeros(n, dtype=np.float32), 1, bits=bits, block=block, beta=0.0, kappa=4.0)
        codes.append(c)
        scales.append(s)
    return codes, scales


def test_decode_w1_is_senders_decompression():
    rng = np.random.default_rng(13)
    for bits, block in [(4, 256), (8, 64)]:
        n = 3 * block + 11
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        err = np.zeros(n, dtype=np.float32)
        c, s = run(g, err, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
        mean = oracle.decode_reduce([c], [s], n, bits=bits, block=block)
        # beta = 0: err holds r = h - d exactly, so d = h - r = g - err
        assert np.array_equal(mean, (g - err).astype(np.float32))
        mean2 = oracle.decode_reduce([c, c], [s, s], n, bits=bits, block=block)
        assert np.array_equal(mean2, mean)


@pytest.mark.parametrize("W", [1, 2, 3, 5, 8, 13, 16])
def test_decode_against_fp64_sum(W):
    rng = np.random.default_rng(100 + W)
    for bits, block in [(4, 256), (8, 128), (4, 64)]:
        n = 4 * block + 29
        codes, scales = _ranks(rng, n, W, bits, block)
        mean, mean64 = oracle.decode_reduce(codes, scales, n, bits=bits, block=block, with_f64=True)
        # independent fp64 evaluation from the unpacked codes
        ds = [unpack_codes(c, bits, n).astype(np.float32) * np.repeat(s, block)[:n] for c, s in zip(codes, scales)]
        ds = [d.astype(np.float32).astype(np.float64) for d in ds]
        exact = np.sum(ds, axis=0) / W
        np.testing.assert_array_equal(mean64, exact) if W <= 2 else np.testing.assert_allclose(mean64, exact, rtol=1e-15, atol=0)
        mag = np.sum(np.abs(ds), axis=0) / W
        tol = (W + 1) * 2.0 ** -24 * mag
        assert np.all(np.abs(mean.astype(np.float64) - exact) <= tol), W
        # rank order matters only at rounding level
        perm = rng.permutation(W)
        meanp = oracle.decode_reduce([codes[i] for i in perm], [scales[i] for i in perm], n, bits=bits, block=block)
        assert np.all(np.abs(meanp.astype(np.float64) - exact) <= tol)


# ---------------------------------------------------------------- Eqn (9): Adam

def test_adam_matches_torch_adamw():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    n, bits, block, W = 3 * 256 + 7, 4, 256, 4
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    p = p0.copy()
    m = np.zeros(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                            weight_decay=hp["weight_decay"], foreach=False, fused=False)
    for t in range(1, 6):
        codes, scales = _ranks(rng, n, W, bits, block)
        g = oracle.decode_reduce(codes, scales, n, bits=bits, block=block)
        # size of the two terms of m: the two forms (explicit sum vs torch's lerp) round
        # differently when they cancel, so compare relative to the terms, not the result
        m_terms = m_terms_acc = (m_terms_acc if t > 1 else 0) + hp["beta1"] * np.abs(m) + (1 - hp["beta1"]) * np.abs(g)
        oracle.adam_step(codes, scales, n, p, m, v, t, bits=bits, block=block, **hp)
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
        ref = tp.detach().numpy()
        st = opt.state[tp]
        np.testing.assert_allclose(p, ref, rtol=1e-6, atol=1e-9)
        # rounding differences carry over from step to step: bound by the summed term sizes
        assert np.all(np.abs(m - st["exp_avg"].numpy()) <= 1e-6 * m_terms + 1e-30)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-5, atol=1e-18)


def test_adam_first_step_is_sign_descent():
    """At t = 1 with bias correction, mh = g and vh = g^2, so the step is lr*g/(|g|+eps)."""
    rng = np.random.default_rng(15)
    n, bits, block = 512, 8, 128
    codes, scales = _ranks(rng, n, 2, bits, block)
    g = oracle.decode_reduce(codes, scales, n, bits=bits, block=block).astype(np.float64)
    p = np.ones(n, dtype=np.float32)
    m = np.zeros(n, dtype=np.float32)
    v = np.zeros(n, dtype=np.float32)
    lr, eps = 1e-2, 1e-12
    oracle.adam_step(codes, scales, n, p, m, v, 1, bits=bits, block=block, lr=lr, beta1=0.9,
                     beta2=0.999, eps=eps)
    want = 1.0 - lr * g / (np.abs(g) + eps)
    np.testing.assert_allclose(p, want, rtol=0, atol=4e-7)


@pytest.mark.parametrize("bits", [4, 8])
def test_tiny_block_whose_inverse_step_overflows(bits):
    """A block with 0 < A_b < qmax/FLT_MAX: s = qmax/A_b is not representable in
    fp32, so the block is treated like an all-zero block: step 0, codes 0, and the
    error range of that zero step (Eqn 7) is {0}, so the stored error is zero.
    Just above the threshold the block quantises normally."""
    qmax = QMAX[bits]
    fmax = float(np.finfo(np.float32).max)
    thresh = qmax / fmax
    block = 64
    tiny = np.float32(thresh * 0.5)
    g = np.zeros(2 * block, dtype=np.float32)
    g[:block:3] = tiny
    g[1:block:5] = -tiny
    big = np.float32(thresh * 4)
    g[block:] = big
    err = np.zeros(2 * block, dtype=np.float32)
    codes, scales = oracle.compress(g, err, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
    assert scales[0] == 0 and not codes[:block * bits // 8].any()
    assert np.all(err[:block] == 0)
    assert scales[1] > 0
    q = unpack_codes(codes, bits, 2 * block)
    assert np.all(q[block:] == qmax)
    qe = np.zeros(2 * block, dtype=np.int8)
    de = np.zeros(2, dtype=np.float32)
    c8, s8 = oracle.compress_e8(g, qe, de, 1, bits=bits, block=block, beta=0.0, kappa=4.0)
    assert np.array_equal(c8, codes) and np.array_equal(s8, scales)
    assert not qe[:block].any()


# ---------------------------------------------------------------- §4 SGD and the bf16 parameter copy

def test_bf16_rounding_matches_torch():
    """The oracle's fp32 -> bf16 rounding (nearest, halves to even) against
    torch's conversion, on random values, exact ties and overflow to inf."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(30)
    x = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32)
    u = x.view(np.uint32)
    ties = ((u & 0xFFFF0000) | 0x8000).view(np.float32)      # exactly halfway
    big = np.array([3.3e38, -3.39e38, np.finfo(np.float32).max], dtype=np.float32)
    vals = np.concatenate([x, ties, big, np.float32([0.0, -0.0, 1e-40, -1e-45])])
    n = vals.size
    codes = [np.zeros(oracle.code_bytes(n, 8, 64), dtype=np.uint8)]
    scales = [np.zeros(oracle.num_blocks(n, 64), dtype=np.float32)]
    p = vals.copy()
    out = np.zeros(n, dtype=np.uint16)
    oracle.sgd_step(codes, scales, n, p, bits=8, block=64, lr=1.0, param_bf16=out)  # g~ = 0: p unchanged
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(p, vals)
    assert np.array_equal(out, want)


def test_sgd_step_closed_form():
    """W = 1, dyadic codes and step: g~ = q*Delta exactly and theta - lr*g~ is exact."""
    n, bits, block = 64, 4, 64
    u = 2.0 ** -10
    q = np.array([4, -4, 2, -1, 7, -8, 0, 3] * 8)
    codes = np.zeros(32, dtype=np.uint8)
    for j in range(0, 64, 2):
        codes[j // 2] = (q[j] & 0xF) | ((q[j + 1] & 0xF) << 4)
    scales = np.array([u], dtype=np.float32)
    p0 = (np.arange(n, dtype=np.float32) - 32) * np.float32(0.25)
    p = p0.copy()
    out = np.zeros(n, dtype=np.uint16)
    oracle.sgd_step([codes], [scales], n, p, bits=bits, block=block, lr=2.0 ** -3, param_bf16=out)
    want = p0.astype(np.float64) - 2.0 ** -3 * q * u
    assert np.array_equal(p.astype(np.float64), want)
    # decode_reduce gives the same g~
    g = oracle.decode_reduce([codes], [scales], n, bits=bits, block=block)
    assert np.array_equal(p, (p0 - np.float32(2.0 ** -3) * g).astype(np.float32))


# ------------------------------------------- rounding paths the readings fix (targeted)

def _rint_even(fr: Fraction) -> int:
    """Nearest integer to an exact rational, halves to even."""
    f = fr.numerator // fr.denominator
    rem = fr - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def _F(x) -> Fraction:
    return Fraction(float(np.float32(x)))


def _inverse_split_case(qmax: int, seed: int):
    """A block maximum A for which RN(qmax/A) and RN(1/RN(A/qmax)) differ, and an
    element h of that block whose code differs between the two (exact rationals)."""
    rng = np.random.default_rng(seed)
    for A in rng.uniform(0.25, 1.0, 4000).astype(np.float32):
        inv = f32_nearest(Fraction(qmax) / _F(A))
        inv_alt = f32_nearest(1 / _F(f32_nearest(_F(A) / qmax)))
        if inv == inv_alt:
            continue
        for k in range(qmax):
            h0 = np.float32(float((Fraction(k) + Fraction(1, 2)) / _F(inv)))
            for d in range(-40, 41):
                h = np.float32(h0)
                h = np.nextafter(h, np.float32(np.inf) if d > 0 else np.float32(-np.inf)) if d else h
                for _ in range(abs(d) - 1):
                    h = np.nextafter(h, np.float32(np.inf) if d > 0 else np.float32(-np.inf))
                if not (0 < h < A):
                    continue
                qa = _rint_even(_F(f32_nearest(_F(h) * _F(inv))))
                qb = _rint_even(_F(f32_nearest(_F(h) * _F(inv_alt))))
                if qa != qb:
                    return A, h, inv, qa, qb
    raise AssertionError("no distinguishing case found")


@pytest.mark.parametrize("bits", [4, 8])
def test_inverse_step_is_rounded_qmax_over_amax(bits):
    """Reading of Eqn (1): codes are rint(h * inv_b) with inv_b = RN(qmax / A_b),
    the IEEE quotient -- not the reciprocal of the stored step.  The case is
    built so that the two inverses round differently and an element's code
    depends on which one is used."""
    qmax = (1 << (bits - 1)) - 1
    A, h, inv, qa, qb = _inverse_split_case(qmax, 40 + bits)
    block = 64
    g = np.zeros(block, dtype=np.float32)
    g[0], g[1] = A, h
    codes, scales = run(g, np.zeros(block, np.float32), 1, bits=bits, block=block, beta=0.5, kappa=4.0)
    q = unpack_codes(codes, bits, block)
    assert scales[0] == f32_nearest(_F(A) / qmax)
    assert q[0] == qmax and q[1] == qa and qa != qb


def test_error_code_inverse_is_kappa_times_inverse_step():
    """Reading of Eqn (7): the 8-bit error code is rint(t * inv_e) with
    inv_e = RN(kappa * inv_b) (s_e = kappa * s), not RN(1 / (Delta_b / kappa)).
    With beta = 0 the stored error before coding is t = r = h - RN(q * Delta_b).
    The element h is placed so that r * inv_e sits at a half-integer k + 1/2
    (k <= 2 keeps |r * inv_b| < 1/2, so q is unchanged) and the two inverses give
    different error codes."""
    kappa = np.float32(6.0)
    qmax, block = 7, 64
    rng = np.random.default_rng(3)

    def nudge(x, steps):
        for _ in range(abs(steps)):
            x = np.nextafter(x, np.float32(np.inf) if steps > 0 else np.float32(-np.inf))
        return x

    found = None
    for A in rng.uniform(0.25, 1.0, 3000).astype(np.float32):
        inv = f32_nearest(Fraction(qmax) / _F(A))
        delta = f32_nearest(_F(A) / qmax)
        inv_e = f32_nearest(_F(kappa) * _F(inv))
        inv_e_alt = f32_nearest(1 / _F(f32_nearest(_F(delta) / _F(kappa))))
        if inv_e == inv_e_alt:
            continue
        for q in (1, 2, 3):
            d = f32_nearest(q * _F(delta))
            for k in (0, 1, 2):
                h0 = np.float32(float(_F(d) + (Fraction(k) + Fraction(1, 2)) / _F(inv_e)))
                for st in range(-48, 49):
                    h = nudge(h0, st)
                    if _rint_even(_F(f32_nearest(_F(h) * _F(inv)))) != q:
                        continue
                    r = f32_nearest(_F(h) - _F(d))
                    ea = _rint_even(_F(f32_nearest(_F(r) * _F(inv_e))))
                    eb = _rint_even(_F(f32_nearest(_F(r) * _F(inv_e_alt))))
                    if ea != eb:
                        found = (A, h, ea, eb)
                        break
                if found:
                    break
            if found:
                break
        if found:
            break
    assert found, "no distinguishing case found"
    A, h, ea, eb = found
    g = np.zeros(block, dtype=np.float32)
    g[0], g[1] = A, h
    qe, de = np.zeros(block, np.int8), np.zeros(1, np.float32)
    oracle.compress_e8(g, qe, de, 1, bits=4, block=block, beta=0.0, kappa=float(kappa))
    assert qe[1] == ea and ea != eb


def test_mean_is_rank_ordered_sum_then_division():
    """Reading of Eqn (8): mean = RN(RN(RN(d_0 + d_1) + d_2) / 3), the fp32 sum in
    rank order divided once -- not the sum of per-rank quotients d_w / 3.  Three
    ranks of one 64-element block whose decoded values make the two orders differ."""
    rng = np.random.default_rng(8)
    W, block, bits = 3, 64, 4
    for _ in range(2000):
        qs = rng.integers(-8, 8, size=W)
        ss = rng.uniform(1e-3, 1.0, size=W).astype(np.float32)
        d = [f32_nearest(int(q) * _F(s)) for q, s in zip(qs, ss)]
        acc = _F(d[0])
        for w in range(1, W):
            acc = _F(f32_nearest(acc + _F(d[w])))
        want = f32_nearest(acc / W)
        acc2 = _F(f32_nearest(_F(d[0]) / W))
        for w in range(1, W):
            acc2 = _F(f32_nearest(acc2 + _F(f32_nearest(_F(d[w]) / W))))
        if want != np.float32(float(acc2)):
            break
    else:
        raise AssertionError("no distinguishing case found")
    codes = []
    for q in qs:
        nib = int(q) & 0xF
        blk = np.zeros(block * bits // 8, dtype=np.uint8)
        blk[0] = nib                                   # element 0 (low nibble); the rest code 0
        codes.append(blk)
    mean = oracle.decode_reduce(codes, [np.array([s], np.float32) for s in ss], block, bits=bits, block=block)
    assert mean[0].view(np.uint32) == want.view(np.uint32)
    assert np.all(mean[1:] == 0)


def test_adam_eps_inside_the_root_closed_form():
    """The pages' form of Eqn (9), eps inside the root: den = sqrt(v_hat + eps).
    A dyadic first step: beta1 = beta2 = 1/2 (both corrections exactly 2), one
    rank with g = 1/2, eps = 3/4, lr = 1/16: m = 1/4, v = 1/8, v_hat = 1/4,
    den = sqrt(1/4 + 3/4) = 1, step = lr * 2 * (1/4) = 1/32, so p = 1 - 1/32
    exactly.  Elements with g = 0 keep p, m and v."""
    bits, block, n = 4, 64, 64
    codes = np.zeros(block * bits // 8, dtype=np.uint8)
    codes[0] = 0x01                                    # element 0: q = 1; the rest q = 0
    scales = np.array([0.5], np.float32)              # g_0 = 1 * 1/2
    p = np.ones(n, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    oracle.adam_step([codes], [scales], n, p, m, v, 1, bits=bits, block=block, lr=1 / 16, beta1=0.5, beta2=0.5,
                     eps=0.75, weight_decay=0.0, bias_correction=True, eps_inside_sqrt=True)
    assert p[0] == np.float32(1 - 1 / 32) and m[0] == np.float32(0.25) and v[0] == np.float32(0.125)
    assert np.all(p[1:] == 1) and np.all(m[1:] == 0) and np.all(v[1:] == 0)


def _f32_sqrt(x: Fraction) -> np.float32:
    """Correctly rounded fp32 square root of an exact non-negative rational: y is
    RN(sqrt(x)) iff x lies between the squares of the midpoints around y (a
    square root of an fp32 value is never exactly a midpoint)."""
    y = np.float32(np.sqrt(float(x)))
    for _ in range(4):
        up, dn = np.nextafter(y, np.float32(np.inf)), np.nextafter(y, np.float32(0))
        hi = (_F(y) + _F(up)) / 2
        lo = (_F(y) + _F(dn)) / 2
        if x > hi * hi:
            y = up
        elif x < lo * lo:
            y = dn
        else:
            return y
    raise AssertionError("square root did not settle")


def test_adam_bias_corrections_folded_into_step_and_denominator():
    """Reading of Eqn (9) (its Adam: the bias corrections of Kingma & Ba's
    Algorithm 1, m_hat = m/(1-b1^t), v_hat = v/(1-b2^t), step lr*m_hat/(sqrt(v_hat)+eps)).
    The oracle folds them: den = RN(RN(sqrt(v))*c2) + eps with c2 = RN(1/sqrt(1-b2^t)),
    step = RN(c1*RN(m/den)) with c1 = RN(lr/(1-b1^t)) -- equal to Algorithm 1 in
    exact arithmetic, different in fp32.  Built in exact rationals with every
    operation rounded to fp32, on an element (t = 3, nonzero state) where the two
    arrangements round to different parameters: the oracle must give the folded one."""
    b1, b2, lr, eps, t = np.float32(0.9), np.float32(0.95), np.float32(1e-3), np.float32(1e-8), 3
    bc1, bc2 = 1.0 - float(b1) ** t, 1.0 - float(b2) ** t        # double, as the constants are formed
    c1, c2 = np.float32(float(lr) / bc1), np.float32(1.0 / np.sqrt(bc2))
    omb1, omb2 = f32_nearest(1 - _F(b1)), f32_nearest(1 - _F(b2))
    R = lambda fr: _F(f32_nearest(fr))                            # round an exact value to fp32
    rng = np.random.default_rng(21)
    for _ in range(5000):
        q = int(rng.integers(-8, 8))
        s = np.float32(rng.uniform(1e-4, 1e-2))
        p0, m0, v0 = (np.float32(x) for x in (rng.uniform(-1, 1), rng.normal(0, 1e-3), rng.uniform(1e-8, 1e-5)))
        g = R(q * _F(s))                                          # one rank: mean = d_0 / 1
        m1 = R(R(_F(b1) * _F(m0)) + R(_F(omb1) * g))
        v1 = R(R(_F(b2) * _F(v0)) + R(_F(omb2) * R(g * g)))
        den = R(R(_F(_f32_sqrt(v1)) * _F(c2)) + _F(eps))
        folded = f32_nearest(_F(p0) - R(_F(c1) * R(m1 / den)))
        mh = R(m1 / _F(np.float32(bc1)))
        vh = R(v1 / _F(np.float32(bc2)))
        den_u = R(_F(_f32_sqrt(vh)) + _F(eps))
        unfolded = f32_nearest(_F(p0) - R(_F(lr) * R(mh / den_u)))
        if folded != unfolded:
            break
    else:
        raise AssertionError("no distinguishing case found")
    bits, block = 4, 64
    codes = np.zeros(block * bits // 8, dtype=np.uint8)
    codes[0] = q & 0xF                                            # element 0 carries q; the rest code 0
    p = np.full(block, p0, np.float32)
    m = np.zeros(block, np.float32)
    v = np.zeros(block, np.float32)
    m[0], v[0] = m0, v0
    oracle.adam_step([codes], [np.array([s], np.float32)], block, p, m, v, t, bits=bits, block=block, lr=float(lr),
                     beta1=float(b1), beta2=float(b2), eps=float(eps), weight_decay=0.0)
    assert m[0] == np.float32(float(m1)) and v[0] == np.float32(float(v1))
    assert p[0].view(np.uint32) == folded.view(np.uint32), (p[0], folded, unfolded)
