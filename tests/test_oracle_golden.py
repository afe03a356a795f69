"""Oracle vs. hand-derived worked examples (tests/golden/worked_examples.json).

Each case was worked out by hand from the rules of "LoCo: Low-Bit
Communication Adaptor for Large-scale Model Training" (§3.1 Eqns 1-3,
§3.2 Eqns 4-7, §3.3 Eqn 8, §4 Eqn 9) with dyadic numbers, so the expected
values are exact in fp32.  They pin rounding (halves to even, negative ties),
saturation, nibble order and sign encoding, padding of a ragged block, the
moving-average weights, the clip bounds, the reset index, the rank average and
the Adam update.
"""
import numpy as np
import pytest

import oracle


def _bf16_bits(x32: np.ndarray) -> np.ndarray:
    u = x32.astype(np.float32).view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "golden values must be exact in bf16"
    return (u >> 16).astype(np.uint16)


def _expected_codes(hexstr, n, bits, block):
    total = oracle.code_bytes(n, bits, block)
    head = bytes.fromhex(hexstr)
    out = np.zeros(total, dtype=np.uint8)
    out[:len(head)] = np.frombuffer(head, dtype=np.uint8)
    return out


def _grad(case):
    g = np.zeros(case["n"], dtype=np.float32)
    head = np.array(case["grad_units_head"], dtype=np.float64) * case["unit"]
    g[:len(head)] = head.astype(np.float32)
    assert np.all(g[:len(head)].astype(np.float64) == head), "golden inputs must be exact in fp32"
    return g


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_compress_worked_examples(golden, dtype):
    for case in golden["compress_cases"]:
        g = _grad(case)
        gin = g if dtype == "f32" else _bf16_bits(g)
        err = np.zeros(case["n"], dtype=np.float32)
        kw = dict(bits=case["bits"], block=case["block"], beta=case["beta"], kappa=case["kappa"],
                  reset_period=case["reset_period"])
        if case["scale_mode"] == "fixed":
            kw["fixed_scale"] = case["fixed_scale"]
        for st in case["steps"]:
            codes, scales = oracle.compress(gin, err, st["step"], **kw)
            exp_codes = _expected_codes(st["codes_head_exact_hex"], case["n"], case["bits"], case["block"])
            assert codes.tobytes().hex() == exp_codes.tobytes().hex(), (case["name"], st["step"])
            np.testing.assert_array_equal(scales, np.float32(st["scale_units"] * case["unit"]),
                                          err_msg=f'{case["name"]} step {st["step"]}')
            exp_err = np.zeros(case["n"], dtype=np.float64)
            head = np.array(st["err_units_head"], dtype=np.float64) * case["unit"]
            exp_err[:len(head)] = head
            assert np.array_equal(err.astype(np.float64), exp_err), (case["name"], st["step"], err[:8] / case["unit"])


def test_decode_worked_examples(golden):
    for case in golden["decode_cases"]:
        n, bits, block, u = case["n"], case["bits"], case["block"], case["unit"]
        codes = [_expected_codes(r["codes_head_exact_hex"], n, bits, block) for r in case["ranks"]]
        nb = oracle.num_blocks(n, block)
        scales = [np.full(nb, np.float32(r["scale_units"] * u), dtype=np.float32) for r in case["ranks"]]
        mean = oracle.decode_reduce(codes, scales, n, bits=bits, block=block)
        head = np.array(case["mean_units_head"], dtype=np.float64) * u
        assert np.array_equal(mean[:len(head)].astype(np.float64), head), (case["name"], mean[:8] / u)
        if case["name"] == "three_ranks_8bit":
            # element 2: sum -5u, divided by 3 and rounded to the nearest fp32 (IEEE division)
            from fractions import Fraction
            exact = Fraction(-5) * Fraction(u) / 3
            got = Fraction(float(mean[2]))
            ulp = Fraction(float(np.spacing(np.float32(abs(float(exact))))))
            assert abs(got - exact) <= ulp / 2
            assert np.all(mean[3:] == 0)


def test_adam_worked_examples(golden):
    for case in golden["adam_cases"]:
        n, bits, block, u = case["n"], case["bits"], case["block"], case["unit"]
        codes = [_expected_codes(case["codes_head_exact_hex"], n, bits, block)]
        scales = [np.full(oracle.num_blocks(n, block), np.float32(case["scale_units"] * u), dtype=np.float32)]
        p = np.array(case["param0"], dtype=np.float32)
        m = np.zeros(n, dtype=np.float32)
        v = np.zeros(n, dtype=np.float32)
        oracle.adam_step(codes, scales, n, p, m, v, case["t"], bits=bits, block=block, lr=case["lr"],
                         beta1=case["beta1"], beta2=case["beta2"], eps=case["eps"],
                         weight_decay=case["weight_decay"], bias_correction=bool(case["bias_correction"]),
                         eps_inside_sqrt=bool(case["eps_inside_sqrt"]))
        assert np.array_equal(p.astype(np.float64), np.array(case["param1"])), (case["name"], p)
        assert np.array_equal(m.astype(np.float64), np.array(case["m1_units"]) * u), (case["name"], m / u)
        assert np.array_equal(v.astype(np.float64), np.array(case["v1_in_2pow_minus20"]) * 2.0 ** -20), case["name"]
