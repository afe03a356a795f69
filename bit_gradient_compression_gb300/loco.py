"""Python binding of libloco (include/loco.h): argument marshalling only.

Every function has the name of the C entry point it calls and does nothing
but turn tensors (or raw integer device addresses) into pointers and sizes,
pick the current torch CUDA stream, and raise ``LocoError`` on a non-OK
status.  All arithmetic runs in the CUDA kernels of ``libloco.so``; there is
no CPU or PyTorch fallback: if the library is missing, importing this module
fails.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libloco.so")

LOCO_OK, LOCO_ERR_INVALID_ARG, LOCO_ERR_UNSUPPORTED, LOCO_ERR_MISALIGNED, LOCO_ERR_CUDA = 0, 1, 2, 3, 4
LOCO_F32, LOCO_BF16 = 0, 1
LOCO_SCALE_ABSMAX, LOCO_SCALE_FIXED = 0, 1
LOCO_MAX_RANKS = 16
LOCO_MAX_N = 1 << 48

EXPORTS = ("loco_num_blocks", "loco_code_bytes", "loco_compress", "loco_compress_e8", "loco_decode_reduce",
           "loco_adam_step", "loco_adam_step_bf16", "loco_sgd_step", "loco_shard_range", "loco_status_string",
           "loco_last_error")


class LocoError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{_status_name(status)}: {message}")


class loco_config(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("block", ctypes.c_int32), ("scale_mode", ctypes.c_int32),
                ("fixed_scale", ctypes.c_float), ("beta", ctypes.c_float), ("err_scale_mult", ctypes.c_float),
                ("reset_period", ctypes.c_int64)]


class loco_adam_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("bias_correction", ctypes.c_int32), ("eps_inside_sqrt", ctypes.c_int32)]


def make_config(bits=4, block=256, beta=0.9, err_scale_mult=4.0, reset_period=0, fixed_scale=None):
    return loco_config(bits, block, LOCO_SCALE_FIXED if fixed_scale is not None else LOCO_SCALE_ABSMAX,
                       float(fixed_scale or 0.0), float(beta), float(err_scale_mult), int(reset_period))


def make_adam(lr=1e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.0, bias_correction=True,
              eps_inside_sqrt=False):
    return loco_adam_hparams(lr, beta1, beta2, eps, weight_decay, int(bias_correction), int(eps_inside_sqrt))


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built: run bit_gradient_compression_gb300.build.build() "
                      "(nvcc, sm_103a); there is no fallback implementation")

lib = ctypes.CDLL(LIB_PATH)
_vp, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
lib.loco_num_blocks.argtypes = [_i64, _i32]
lib.loco_num_blocks.restype = _i64
lib.loco_code_bytes.argtypes = [_i64, _i32, _i32]
lib.loco_code_bytes.restype = _i64
lib.loco_compress.argtypes = [ctypes.POINTER(loco_config), _vp, _i32, _vp, _i64, _i64, _vp, _vp, _vp]
lib.loco_compress.restype = ctypes.c_int
lib.loco_compress_e8.argtypes = [ctypes.POINTER(loco_config), _vp, _i32, _vp, _vp, _i64, _i64, _vp, _vp, _vp]
lib.loco_compress_e8.restype = ctypes.c_int
lib.loco_decode_reduce.argtypes = [ctypes.POINTER(loco_config), _vp, _vp, _i32, _i64, _vp, _vp]
lib.loco_decode_reduce.restype = ctypes.c_int
lib.loco_adam_step.argtypes = [ctypes.POINTER(loco_config), _vp, _vp, _i32, _i64, _vp, _vp, _vp,
                               ctypes.POINTER(loco_adam_hparams), _i64, _vp]
lib.loco_adam_step.restype = ctypes.c_int
lib.loco_adam_step_bf16.argtypes = [ctypes.POINTER(loco_config), _vp, _vp, _i32, _i64, _vp, _vp, _vp, _vp,
                                    ctypes.POINTER(loco_adam_hparams), _i64, _vp]
lib.loco_adam_step_bf16.restype = ctypes.c_int
lib.loco_sgd_step.argtypes = [ctypes.POINTER(loco_config), _vp, _vp, _i32, _i64, _vp, _vp, ctypes.c_float, _vp]
lib.loco_sgd_step.restype = ctypes.c_int
lib.loco_shard_range.argtypes = [_i64, _i32, _i32, _i32, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
lib.loco_shard_range.restype = ctypes.c_int
lib.loco_status_string.argtypes = [ctypes.c_int]
lib.loco_status_string.restype = ctypes.c_char_p
lib.loco_last_error.argtypes = []
lib.loco_last_error.restype = ctypes.c_char_p


def _status_name(s: int) -> str:
    return lib.loco_status_string(s).decode()


def _check(status: int):
    if status != LOCO_OK:
        raise LocoError(status, lib.loco_last_error().decode())


def _addr(x) -> int:
    """Device address of a tensor (must be contiguous) or an integer address."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("tensors passed to libloco must be contiguous")
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _grad_dtype(grad, grad_dtype):
    if grad_dtype is not None:
        return grad_dtype
    import torch
    if grad.dtype == torch.bfloat16:
        return LOCO_BF16
    if grad.dtype == torch.float32:
        return LOCO_F32
    raise ValueError(f"gradient dtype {grad.dtype} is not supported (float32 or bfloat16)")


def loco_num_blocks(n: int, block: int) -> int:
    return lib.loco_num_blocks(n, block)


def loco_code_bytes(n: int, bits: int, block: int) -> int:
    return lib.loco_code_bytes(n, bits, block)


def loco_compress(cfg: loco_config, grad, err, step: int, codes, scales, *, n: int | None = None,
                  grad_dtype: int | None = None, stream=None):
    """Sender step (compensate, quantise, pack, error update) on one bucket."""
    if n is None:
        n = grad.numel()
    _check(lib.loco_compress(ctypes.byref(cfg), _addr(grad), _grad_dtype(grad, grad_dtype), _addr(err),
                             n, step, _addr(codes), _addr(scales), _stream(stream)))


def loco_compress_e8(cfg: loco_config, grad, err_codes, err_steps, step: int, codes, scales, *,
                     n: int | None = None, grad_dtype: int | None = None, stream=None):
    """Sender step with the error kept as int8 codes + one step per block (updated in place)."""
    if n is None:
        n = grad.numel()
    _check(lib.loco_compress_e8(ctypes.byref(cfg), _addr(grad), _grad_dtype(grad, grad_dtype), _addr(err_codes),
                                _addr(err_steps), n, step, _addr(codes), _addr(scales), _stream(stream)))


def _rank_arrays(codes, scales):
    W = len(codes)
    if len(scales) != W:
        raise ValueError("codes and scales must list the same ranks")
    ca = (ctypes.c_void_p * max(W, 1))(*[_addr(c) for c in codes])
    sa = (ctypes.c_void_p * max(W, 1))(*[_addr(s) for s in scales])
    return W, ca, sa


def loco_decode_reduce(cfg: loco_config, codes, scales, n: int, mean, *, stream=None):
    """Average of W ranks' decoded buckets (fp32), written to mean."""
    W, ca, sa = _rank_arrays(codes, scales)
    _check(lib.loco_decode_reduce(ctypes.byref(cfg), ca, sa, W, n, _addr(mean), _stream(stream)))


def loco_adam_step(cfg: loco_config, codes, scales, n: int, param, m, v, hp: loco_adam_hparams, t: int, *,
                   stream=None):
    """Decode-reduce fused with one Adam(W) update of param, m, v (in place)."""
    W, ca, sa = _rank_arrays(codes, scales)
    _check(lib.loco_adam_step(ctypes.byref(cfg), ca, sa, W, n, _addr(param), _addr(m), _addr(v),
                              ctypes.byref(hp), t, _stream(stream)))


def loco_adam_step_bf16(cfg: loco_config, codes, scales, n: int, param, m, v, param_bf16, hp: loco_adam_hparams,
                        t: int, *, stream=None):
    """loco_adam_step that also writes bf16(param) into param_bf16."""
    W, ca, sa = _rank_arrays(codes, scales)
    _check(lib.loco_adam_step_bf16(ctypes.byref(cfg), ca, sa, W, n, _addr(param), _addr(m), _addr(v),
                                   _addr(param_bf16), ctypes.byref(hp), t, _stream(stream)))


def loco_sgd_step(cfg: loco_config, codes, scales, n: int, param, lr: float, *, param_bf16=None, stream=None):
    """Decode-reduce fused with one LoCo-SGD step (param -= lr * mean), optional bf16 copy."""
    W, ca, sa = _rank_arrays(codes, scales)
    _check(lib.loco_sgd_step(ctypes.byref(cfg), ca, sa, W, n, _addr(param), _addr(param_bf16), float(lr),
                             _stream(stream)))


def loco_shard_range(n: int, block: int, W: int, j: int) -> tuple[int, int]:
    """Element range [lo, hi) of shard j of W (the sharded receiver's split of a bucket)."""
    lo, hi = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.loco_shard_range(n, block, W, j, ctypes.byref(lo), ctypes.byref(hi)))
    return lo.value, hi.value
