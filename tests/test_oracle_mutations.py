"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/loco_oracle.c (a dropped
term, a swapped weight, a wrong sign or index, the wrong rounding rule, ...),
builds it, and runs the CPU pin tests against it in a subprocess: at least one
pin must fail.  The unmodified source must pass the same tests.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "loco_oracle.c")
PIN_TESTS = ["tests/test_oracle_golden.py", "tests/test_oracle_pins.py", "tests/test_oracle_e8.py"]

# (name, text in the source, replacement, occurrence to replace (0 = all))
MUTATIONS = [
    ("round half away from zero", "return (int)nearbyintf(x);", "return (int)roundf(x);", 0),
    ("compensation term dropped", "h[j] = g + err[lo + j];", "h[j] = g;", 0),
    ("beta weights swapped", "float t1 = beta * prev;", "float t1 = one_minus_beta * prev;", 1),
    ("residual sign flipped", "float r = h[j] - d;", "float r = d - h[j];", 1),
    ("nibble order swapped", "if (j % 2 == 0)\n      blk[j / 2] = (uint8_t)((blk[j / 2] & 0xF0) | nib);",
     "if (j % 2 == 1)\n      blk[j / 2] = (uint8_t)((blk[j / 2] & 0xF0) | nib);", 0),
    ("clip bound off by one code", "const float e_lo = -128.0f * delta_e;", "const float e_lo = -127.0f * delta_e;", 0),
    ("reset one step late", "(step % reset_period == 0)", "((step - 1) % reset_period == 0)", 1),
    ("scale uses qmax+1", "delta = amax / qmax;", "delta = amax / (qmax + 1.0f);", 1),
    ("last rank dropped from the mean", "for (int w = 0; w < W; ++w) {\n      int q = get_code(codes[w] + b * bytes_per_block, bits, j);\n      float d = (float)q * scales[w][b];\n      acc = (w == 0) ? d : acc + d;\n      acc64 += (double)d;",
     "for (int w = 0; w < W - (W > 1); ++w) {\n      int q = get_code(codes[w] + b * bytes_per_block, bits, j);\n      float d = (float)q * scales[w][b];\n      acc = (w == 0) ? d : acc + d;\n      acc64 += (double)d;", 0),
    ("Adam first moment weights swapped", "float mi = beta1 * m[i];\n    float mg = omb1 * g;",
     "float mi = omb1 * m[i];\n    float mg = beta1 * g;", 0),
    ("Adam bias correction of v dropped", "c2 = eps_inside_sqrt ? (float)(1.0 / bc2) : (float)(1.0 / sqrt(bc2));",
     "c2 = 1.0f;", 0),
    ("8-bit error scale divides by kappa", "float inv_e = kappa * inv;", "float inv_e = inv / kappa;", 0),
    ("8-bit error not decompressed", "prev[j] = (float)err_codes[lo + j] * de_prev;", "prev[j] = (float)err_codes[lo + j];", 0),
    ("bf16 truncation instead of rounding", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;", 0),
    ("SGD step sign flipped", "float p = param[i] - step;", "float p = param[i] + step;", 0),
    ("Adam eps dropped (eps outside the root)", "den = rs + eps;", "den = rs;", 0),
    ("decoupled weight decay dropped", "p = p - decay;", "p = p - 0.0f * decay;", 0),
    ("Adam bias corrections unfolded (m_hat, v_hat formed first)",
     "      float r = sqrtf(vi);\n      float rs = r * c2;\n      den = rs + eps;\n    }\n    float ratio = mi / den;\n"
     "    float step = c1 * ratio;",
     "      float vh = vi / (float)(1.0 - pow((double)beta2, (double)t));\n      float r = sqrtf(vh);\n"
     "      den = r + eps;\n    }\n    float ratio = (mi / (float)(1.0 - pow((double)beta1, (double)t))) / den;\n"
     "    float step = lr * ratio;", 0),
    ("clip upper bound 128 codes", "const float e_hi = 127.0f * delta_e;", "const float e_hi = 128.0f * delta_e;", 0),
    ("padding codes nonzero", "put_code(blk, bits, j, 0);", "put_code(blk, bits, j, 1);", 0),
    ("int8 error decoded with a neighbouring block's step", "const float de_prev = err_steps[b];",
     "const float de_prev = err_steps[b > b0 ? b - 1 : b];", 0),
    ("every rank decoded with rank 0's step", "float d = (float)q * scales[w][b];", "float d = (float)q * scales[0][b];", 0),
    ("v accumulates |g| instead of g*g", "float gg = g * g;", "float gg = g < 0 ? -g : g;", 0),
    ("fixed step s instead of 1/s", "delta = 1.0f / fixed_scale;", "delta = fixed_scale;", 0),
    ("rank sum in reverse order",
     "int q = get_code(codes[w] + b * bytes_per_block, bits, j);\n      float d = (float)q * scales[w][b];\n      acc = (w == 0) ? d : acc + d;\n      acc64 += (double)d;",
     "int q = get_code(codes[W - 1 - w] + b * bytes_per_block, bits, j);\n      float d = (float)q * scales[W - 1 - w][b];\n      acc = (w == 0) ? d : acc + d;\n      acc64 += (double)d;", 0),
    ("mean divided per term", "acc = (w == 0) ? d : acc + d;\n      acc64 += (double)d;\n    }\n    mean[i] = acc / (float)W;",
     "acc = (w == 0) ? d / (float)W : acc + d / (float)W;\n      acc64 += (double)d;\n    }\n    mean[i] = acc;", 0),
    ("Adam m bias correction uses beta2", "c1 = (float)((double)lr / bc1);", "c1 = (float)((double)lr / bc2);", 0),
    ("inverse step as 1/delta", "inv = (amax == 0.0f) ? 0.0f : qmax / amax;",
     "inv = (amax == 0.0f) ? 0.0f : 1.0f / (amax / qmax);", 0),
    ("int8 error inverse as 1/(delta/kappa)", "float inv_e = kappa * inv;",
     "float inv_e = (de_new == 0.0f) ? 0.0f : 1.0f / de_new;", 0),
    ("bf16 ties rounded up", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;", 0),
    ("absmax skips the last element", "float amax = 0.0f;\n      for (int64_t j = 0; j < cnt; ++j) {",
     "float amax = 0.0f;\n      for (int64_t j = 0; j < cnt - 1; ++j) {", 0),
    ("m accumulates g*g", "float mg = omb1 * g;", "float mg = omb1 * (g * g);", 0),
    ("reset applied before compensation", "h[j] = g + err[lo + j];", "h[j] = g + (reset ? 0.0f : err[lo + j]);", 0),
    ("eps dropped inside the root", "float s = vs + eps;", "float s = vs;", 0),
    ("weight decay without lr", "const float lr_wd = lr * wd;", "const float lr_wd = wd;", 0),
    ("nibbles decoded unsigned", "return nib >= 8 ? nib - 16 : nib;", "return nib;", 0),
    ("symmetric clamp at -qmax", "float qmin = -(float)(1 << (bits - 1));", "float qmin = -qmax;", 0),
    ("int8 error coded with the gradient code width", "int qe = round_pbit(xe, 8);", "int qe = round_pbit(xe, bits);", 0),
    ("int8 error not reset", "if (reset) qe = 0;", "if (0) qe = 0;", 0),
    ("8-bit codes decoded unsigned", "if (bits == 8) return (int)(int8_t)blk[j];", "if (bits == 8) return (int)blk[j];", 0),
    ("8-bit code sign bit dropped", "blk[j] = (uint8_t)(q & 0xFF);", "blk[j] = (uint8_t)(q & 0x7F);", 0),
    ("bias correction at t+1", "double bc1 = 1.0 - pow((double)beta1, (double)t);",
     "double bc1 = 1.0 - pow((double)beta1, (double)(t + 1));", 0),
    ("v correction without its square root",
     "c2 = eps_inside_sqrt ? (float)(1.0 / bc2) : (float)(1.0 / sqrt(bc2));", "c2 = (float)(1.0 / bc2);", 0),
]


def _build(src_text, out_dir, name):
    import oracle
    c = os.path.join(out_dir, f"{name}.c")
    so = os.path.join(out_dir, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.check_call(["gcc", *oracle.CFLAGS, c, "-o", so, "-lm"])
    return so


def _run_pins(so):
    env = dict(os.environ, LOCO_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "not gpu", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def _mutate(text, old, new, occurrence):
    assert old in text, f"mutation anchor not found: {old[:60]!r}"
    if occurrence == 0:
        return text.replace(old, new)
    idx = -1
    for _ in range(occurrence):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.fixture(scope="module")
def outcomes(source, tmp_path_factory):
    """Pin-run exit status of the unmodified copy and of every mutant, computed
    concurrently (each is an independent gcc build plus a pytest subprocess)."""
    import concurrent.futures as cf
    d = str(tmp_path_factory.mktemp("mutants"))
    jobs = {"unmodified": source}
    for i, (name, old, new, occurrence) in enumerate(MUTATIONS):
        jobs[name] = _mutate(source, old, new, occurrence)

    def one(item):
        k, (name, text) = item
        return name, _run_pins(_build(text, d, f"loco_oracle_{k}"))

    workers = max(1, min(8, (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 4)))
    with cf.ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(one, enumerate(jobs.items())))


def test_unmodified_oracle_passes(outcomes):
    rc, out = outcomes["unmodified"]
    assert rc == 0, out


@pytest.mark.parametrize("name,old,new,occurrence", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(outcomes, name, old, new, occurrence):
    rc, out = outcomes[name]
    assert rc != 0, f"no pin caught the planted mistake: {name}\n{out}"
