"""CPU oracle of the LoCo hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product path (the CUDA
library and its binding) never calls it and never falls back to it.

The arithmetic lives in ``loco_oracle.c`` (plain C, fp32, no FMA
contraction); this module compiles it with gcc and exposes numpy-level
wrappers.  Method: "LoCo: Low-Bit Communication Adaptor for Large-scale Model
Training" (arXiv 2407.04480), §3.1-§3.3 and §4.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
hand-derived worked examples (``tests/golden/``), closed forms, invariants and
brute force; see that file for which pin covers which step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "loco_oracle.c")
# A test may point the oracle at another build of this source (the mutation
# test does, to check that the pins catch planted mistakes).
_LIB = os.environ.get("LOCO_ORACLE_LIB") or os.path.join(_HERE, "libloco_oracle.so")

# -ffp-contract=off: every product and sum is its own rounded fp32 operation.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libloco_oracle.so`` (gcc)."""
    if os.environ.get("LOCO_ORACLE_LIB"):
        return _LIB
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            vp = ctypes.c_void_p
            lib.oracle_compress.argtypes = [i32, i32, i32, f32, f32, f32, i64,
                                            vp, i32, vp, i64, i64, vp, vp, i64, i64]
            lib.oracle_compress.restype = None
            lib.oracle_decode_reduce.argtypes = [i32, i32, vp, vp, i32, i64, i64, vp, vp]
            lib.oracle_decode_reduce.restype = None
            lib.oracle_adam_step.argtypes = [i32, i32, vp, vp, i32, i64, i64, vp, vp, vp, vp,
                                             f32, f32, f32, f32, f32, i32, i32, i64]
            lib.oracle_adam_step.restype = None
            lib.oracle_compress_e8.argtypes = [i32, i32, i32, f32, f32, f32, i64,
                                               vp, i32, vp, vp, i64, i64, vp, vp, i64, i64]
            lib.oracle_compress_e8.restype = None
            lib.oracle_sgd_step.argtypes = [i32, i32, vp, vp, i32, i64, i64, vp, vp, f32]
            lib.oracle_sgd_step.restype = None
            _lib = lib
    return _lib


def num_blocks(n: int, block: int) -> int:
    return (n + block - 1) // block


def code_bytes(n: int, bits: int, block: int) -> int:
    return num_blocks(n, block) * block * bits // 8


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ranges(total: int, threads: int):
    threads = max(1, min(threads, total))
    step = (total + threads - 1) // threads
    return [(s, min(s + step, total)) for s in range(0, total, step)]


def _run(fn, ranges):
    if len(ranges) == 1:
        fn(*ranges[0])
        return
    # ctypes releases the GIL during foreign calls, so plain threads run the
    # C loops in parallel on disjoint ranges.
    ts = [threading.Thread(target=fn, args=r) for r in ranges]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


def compress(grad: np.ndarray, err: np.ndarray, step: int, *, bits: int, block: int,
             beta: float, kappa: float, reset_period: int = 0, fixed_scale: float | None = None,
             threads: int = 1, codes: np.ndarray | None = None, scales: np.ndarray | None = None):
    """One LoCo sender step (§3.1 Eqns 1-3, §3.2 Eqns 4-7) on a flat bucket.

    grad: float32 array, or uint16 array holding bf16 bit patterns.
    err:  float32 array, UPDATED IN PLACE (e_{k-1} -> e_k).
    Returns (codes uint8 [code_bytes], scales float32 [nb]).
    """
    lib = _load()
    n = grad.size
    assert err.dtype == np.float32 and err.size == n
    if grad.dtype == np.uint16:
        is_bf16 = 1
    else:
        assert grad.dtype == np.float32
        is_bf16 = 0
    nb = num_blocks(n, block)
    if codes is None:
        codes = np.zeros(code_bytes(n, bits, block), dtype=np.uint8)
    if scales is None:
        scales = np.zeros(nb, dtype=np.float32)
    fixed = fixed_scale is not None
    fs = float(fixed_scale) if fixed else 0.0
    gp, ep, cp, sp = _ptr(grad), _ptr(err), _ptr(codes), _ptr(scales)

    def fn(b0, b1):
        lib.oracle_compress(bits, block, int(fixed), fs, float(beta), float(kappa), int(reset_period),
                            gp, is_bf16, ep, n, int(step), cp, sp, b0, b1)

    if nb:
        _run(fn, _ranges(nb, threads))
    return codes, scales


def compress_e8(grad: np.ndarray, err_codes: np.ndarray, err_steps: np.ndarray, step: int, *, bits: int,
                block: int, beta: float, kappa: float, reset_period: int = 0, fixed_scale: float | None = None,
                threads: int = 1, codes: np.ndarray | None = None, scales: np.ndarray | None = None):
    """LoCo sender step with the error stored as int8 codes + per-block step (§3.2 Eqn 7).

    err_codes (int8 [n]) and err_steps (float32 [nb]) are UPDATED IN PLACE; start from zeros.
    Returns (codes uint8 [code_bytes], scales float32 [nb]).
    """
    lib = _load()
    n = grad.size
    nb = num_blocks(n, block)
    assert err_codes.dtype == np.int8 and err_codes.size == n
    assert err_steps.dtype == np.float32 and err_steps.size == nb
    is_bf16 = 1 if grad.dtype == np.uint16 else 0
    if not is_bf16:
        assert grad.dtype == np.float32
    if codes is None:
        codes = np.zeros(code_bytes(n, bits, block), dtype=np.uint8)
    if scales is None:
        scales = np.zeros(nb, dtype=np.float32)
    fixed = fixed_scale is not None
    fs = float(fixed_scale) if fixed else 0.0
    gp, qp, sp_, cp, scp = _ptr(grad), _ptr(err_codes), _ptr(err_steps), _ptr(codes), _ptr(scales)

    def fn(b0, b1):
        lib.oracle_compress_e8(bits, block, int(fixed), fs, float(beta), float(kappa), int(reset_period),
                               gp, is_bf16, qp, sp_, n, int(step), cp, scp, b0, b1)

    if nb:
        _run(fn, _ranges(nb, threads))
    return codes, scales


def _ptr_array(arrs, ctype):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


def decode_reduce(codes_list, scales_list, n: int, *, bits: int, block: int,
                  with_f64: bool = False, threads: int = 1):
    """Average of W ranks' decompressed codes (§3.3 Eqn 8), fp32, rank order."""
    lib = _load()
    W = len(codes_list)
    assert W == len(scales_list) and W >= 1
    mean = np.empty(n, dtype=np.float32)
    mean64 = np.empty(n, dtype=np.float64) if with_f64 else None
    cpa = _ptr_array(codes_list, ctypes.c_uint8)
    spa = _ptr_array(scales_list, ctypes.c_float)
    mp = _ptr(mean)
    m64p = _ptr(mean64) if with_f64 else None

    def fn(i0, i1):
        lib.oracle_decode_reduce(bits, block, cpa, spa, W, i0, i1, mp, m64p)

    if n:
        _run(fn, _ranges(n, threads))
    return (mean, mean64) if with_f64 else mean


def adam_step(codes_list, scales_list, n: int, param: np.ndarray, m: np.ndarray, v: np.ndarray,
              t: int, *, bits: int, block: int, lr: float, beta1: float, beta2: float,
              eps: float, weight_decay: float = 0.0, bias_correction: bool = True,
              eps_inside_sqrt: bool = False, param_bf16: np.ndarray | None = None, threads: int = 1):
    """Eqn 8 average fed to one Adam(W) step (§4 Eqn 9); param, m, v updated in place.
    param_bf16 (uint16 [n], optional) receives the updated param rounded to bf16."""
    lib = _load()
    W = len(codes_list)
    for a in (param, m, v):
        assert a.dtype == np.float32 and a.size == n
    if param_bf16 is not None:
        assert param_bf16.dtype == np.uint16 and param_bf16.size == n
    cpa = _ptr_array(codes_list, ctypes.c_uint8)
    spa = _ptr_array(scales_list, ctypes.c_float)
    pp, mp, vp = _ptr(param), _ptr(m), _ptr(v)
    bp = _ptr(param_bf16) if param_bf16 is not None else None

    def fn(i0, i1):
        lib.oracle_adam_step(bits, block, cpa, spa, W, i0, i1, pp, mp, vp, bp,
                             float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                             int(bias_correction), int(eps_inside_sqrt), int(t))

    if n:
        _run(fn, _ranges(n, threads))


def sgd_step(codes_list, scales_list, n: int, param: np.ndarray, *, bits: int, block: int, lr: float,
             param_bf16: np.ndarray | None = None, threads: int = 1):
    """Eqn 8 average fed to one LoCo-SGD step (§4): param -= lr * g~ (in place)."""
    lib = _load()
    W = len(codes_list)
    assert param.dtype == np.float32 and param.size == n
    if param_bf16 is not None:
        assert param_bf16.dtype == np.uint16 and param_bf16.size == n
    cpa = _ptr_array(codes_list, ctypes.c_uint8)
    spa = _ptr_array(scales_list, ctypes.c_float)
    pp = _ptr(param)
    bp = _ptr(param_bf16) if param_bf16 is not None else None

    def fn(i0, i1):
        lib.oracle_sgd_step(bits, block, cpa, spa, W, i0, i1, pp, bp, float(lr))

    if n:
        _run(fn, _ranges(n, threads))
