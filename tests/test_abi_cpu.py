"""libloco without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bit_gradient_compression_gb300 import build
    build.build()
    from bit_gradient_compression_gb300 import loco
    return loco


def header_functions():
    src = open(os.path.join(ROOT, "include", "loco.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(loco_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = header_functions()
    assert len(names) >= 7
    raw = ctypes.CDLL(L.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), name
    assert set(names) == set(L.EXPORTS)


def _defined_dynamic_symbols(path):
    """Names of the global/weak symbols an ELF64 little-endian shared object defines (.dynsym)."""
    import struct
    data = open(path, "rb").read()
    assert data[:4] == b"\x7fELF" and data[4] == 2 and data[5] == 1, "ELF64 little-endian expected"
    shoff, = struct.unpack_from("<Q", data, 0x28)
    shentsize, shnum = struct.unpack_from("<HH", data, 0x3A)
    secs = [struct.unpack_from("<IIQQQQIIQQ", data, shoff + i * shentsize) for i in range(shnum)]
    names = set()
    for sec in secs:
        if sec[1] != 11:  # SHT_DYNSYM
            continue
        strtab = secs[sec[6]]
        off, size, entsize = sec[4], sec[5], sec[9]
        for k in range(1, size // entsize):
            st_name, st_info, _, st_shndx, _, _ = struct.unpack_from("<IBBHQQ", data, off + k * entsize)
            if st_shndx == 0 or (st_info >> 4) not in (1, 2):  # undefined, or not GLOBAL/WEAK
                continue
            s0 = strtab[4] + st_name
            names.add(data[s0:data.index(b"\0", s0)].decode())
    return names


def test_exports_nothing_else(L):
    """Only the header's entry points are visible: kernels, helpers and the
    static CUDA runtime stay hidden, so nothing can be interposed between the
    library and other CUDA code (or another build of itself) in one process."""
    assert _defined_dynamic_symbols(L.LIB_PATH) == set(header_functions())


def test_sizes(L):
    assert L.loco_num_blocks(0, 256) == 0
    assert L.loco_num_blocks(1, 256) == 1
    assert L.loco_num_blocks(257, 256) == 2
    assert L.loco_code_bytes(257, 4, 256) == 256
    assert L.loco_code_bytes(257, 8, 64) == 5 * 64
    n7b = 6_738_415_616
    assert L.loco_num_blocks(n7b, 256) == 26_321_936
    assert L.loco_code_bytes(n7b, 4, 256) == n7b // 2
    assert L.loco_code_bytes(1 << 31, 8, 64) == 1 << 31
    # the largest accepted bucket, and beyond it (no int64 overflow anywhere)
    assert L.loco_num_blocks(L.LOCO_MAX_N, 64) == L.LOCO_MAX_N // 64
    assert L.loco_code_bytes(L.LOCO_MAX_N, 8, 64) == L.LOCO_MAX_N
    for n in (L.LOCO_MAX_N + 1, 1 << 62, 2 ** 63 - 1):
        assert L.loco_num_blocks(n, 256) == 0 and L.loco_code_bytes(n, 8, 256) == 0


def _compress(L, cfg, **kw):
    a = dict(grad=0x10000, err=0x20000, step=1, codes=0x30000, scales=0x40000, n=1000, grad_dtype=0, stream=0)
    a.update(kw)
    return L.loco_compress(cfg, a["grad"], a["err"], a["step"], a["codes"], a["scales"], n=a["n"],
                           grad_dtype=a["grad_dtype"], stream=a["stream"])


def _status(L, fn):
    try:
        fn()
    except L.LocoError as e:
        return e.status
    return L.LOCO_OK


def test_argument_errors(L):
    ok = L.make_config()
    st = lambda **kw: _status(L, lambda: _compress(L, kw.pop("cfg", ok), **kw))
    assert st(cfg=L.make_config(bits=3)) == L.LOCO_ERR_UNSUPPORTED
    assert st(cfg=L.make_config(block=32)) == L.LOCO_ERR_UNSUPPORTED
    assert st(cfg=L.make_config(block=512)) == L.LOCO_ERR_UNSUPPORTED
    assert st(grad_dtype=7) == L.LOCO_ERR_UNSUPPORTED
    assert st(cfg=L.make_config(beta=1.5)) == L.LOCO_ERR_INVALID_ARG
    assert st(cfg=L.make_config(beta=-0.1)) == L.LOCO_ERR_INVALID_ARG
    assert st(cfg=L.make_config(beta=float("nan"))) == L.LOCO_ERR_INVALID_ARG
    assert st(cfg=L.make_config(err_scale_mult=0.0)) == L.LOCO_ERR_INVALID_ARG
    assert st(cfg=L.make_config(fixed_scale=-1.0)) == L.LOCO_ERR_INVALID_ARG
    assert st(cfg=L.make_config(reset_period=-1)) == L.LOCO_ERR_INVALID_ARG
    assert st(n=-1) == L.LOCO_ERR_INVALID_ARG
    assert st(n=L.LOCO_MAX_N + 1) == L.LOCO_ERR_INVALID_ARG
    assert st(n=2 ** 63 - 1) == L.LOCO_ERR_INVALID_ARG
    assert st(step=0) == L.LOCO_ERR_INVALID_ARG
    assert st(grad=0) == L.LOCO_ERR_INVALID_ARG
    assert st(err=0) == L.LOCO_ERR_INVALID_ARG
    assert st(grad=0x10001) == L.LOCO_ERR_MISALIGNED
    assert st(codes=0x30008) == L.LOCO_ERR_MISALIGNED
    assert st(scales=0x40002) == L.LOCO_ERR_MISALIGNED
    assert st(scales=0x40004) == L.LOCO_ERR_MISALIGNED
    assert st(scales=0x40008) == L.LOCO_ERR_MISALIGNED
    # n == 0 is an empty, successful call (nothing is launched or dereferenced)
    assert st(n=0, grad=0, err=0, codes=0, scales=0) == L.LOCO_OK
    # non-device memory is refused before any launch (here: no driver at all)
    assert st() == L.LOCO_ERR_INVALID_ARG
    assert L.lib.loco_last_error().decode() != ""


def test_rank_argument_errors(L):
    cfg = L.make_config()
    hp = L.make_adam()
    dr = lambda W, n=100: _status(L, lambda: L.loco_decode_reduce(cfg, [0x1000] * W, [0x2000] * W, n, 0x3000, stream=0))
    assert dr(0) == L.LOCO_ERR_INVALID_ARG
    assert dr(17) == L.LOCO_ERR_UNSUPPORTED
    assert dr(4, n=-5) == L.LOCO_ERR_INVALID_ARG
    assert dr(4, n=2 ** 62) == L.LOCO_ERR_INVALID_ARG
    assert dr(4, n=0) == L.LOCO_OK
    assert _status(L, lambda: L.loco_decode_reduce(cfg, [0x1001], [0x2000], 10, 0x3000, stream=0)) == L.LOCO_ERR_MISALIGNED
    ad = lambda W, t=1, hp=hp: _status(L, lambda: L.loco_adam_step(cfg, [0x1000] * W, [0x2000] * W, 100, 0x3000,
                                                                  0x4000, 0x5000, hp, t, stream=0))
    assert ad(0) == L.LOCO_ERR_INVALID_ARG
    assert ad(17) == L.LOCO_ERR_UNSUPPORTED
    assert ad(2, t=0) == L.LOCO_ERR_INVALID_ARG
    assert _status(L, lambda: L.loco_adam_step(cfg, [0x1000] * 2, [0x2000] * 2, 2 ** 62, 0x3000, 0x4000, 0x5000,
                                               hp, 1, stream=0)) == L.LOCO_ERR_INVALID_ARG
    assert _status(L, lambda: L.loco_sgd_step(cfg, [0x1000] * 2, [0x2000] * 2, 2 ** 62, 0x3000, 0.1,
                                              stream=0)) == L.LOCO_ERR_INVALID_ARG
    assert ad(2, hp=L.make_adam(beta1=1.0)) == L.LOCO_ERR_INVALID_ARG
    assert ad(2, hp=L.make_adam(eps=-1.0)) == L.LOCO_ERR_INVALID_ARG
    assert ad(2, hp=L.make_adam(lr=float("inf"))) == L.LOCO_ERR_INVALID_ARG


def test_scales_must_be_16_byte_aligned(L):
    """The receivers stage each rank's steps with 16-byte copies, so a scales
    pointer at 4, 8 or 12 bytes past a 16-byte boundary is refused on the host
    (nothing is launched) by every entry point that reads or writes steps."""
    cfg = L.make_config()
    hp = L.make_adam()
    st = lambda fn: _status(L, fn)
    for bad in (0x40004, 0x40008, 0x4000C):
        # rank 1 of 3 carries the misaligned steps
        sc = [0x40000, bad, 0x50000]
        assert st(lambda: L.loco_decode_reduce(cfg, [0x1000] * 3, sc, 100, 0x3000, stream=0)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_adam_step(cfg, [0x1000] * 3, sc, 100, 0x3000, 0x4000, 0x5000, hp, 1,
                                           stream=0)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_adam_step_bf16(cfg, [0x1000] * 3, sc, 100, 0x3000, 0x4000, 0x5000, 0x6000, hp, 1,
                                                stream=0)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_sgd_step(cfg, [0x1000] * 3, sc, 100, 0x3000, 0.1, stream=0)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_sgd_step(cfg, [0x1000] * 3, sc, 100, 0x3000, 0.1, param_bf16=0x6000,
                                          stream=0)) == L.LOCO_ERR_MISALIGNED
        # the sender's outputs: steps and the int8 error's per-block steps
        assert st(lambda: _compress(L, cfg, scales=bad)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_compress_e8(cfg, 0x10000, 0x20000, bad, 1, 0x30000, 0x40000, n=1000,
                                             grad_dtype=0, stream=0)) == L.LOCO_ERR_MISALIGNED
        assert st(lambda: L.loco_compress_e8(cfg, 0x10000, 0x20000, 0x60000, 1, 0x30000, bad, n=1000,
                                             grad_dtype=0, stream=0)) == L.LOCO_ERR_MISALIGNED
    assert "16-byte aligned" in L.lib.loco_last_error().decode()


def test_status_strings(L):
    for s in range(5):
        assert L.lib.loco_status_string(s).decode().startswith("LOCO_")


def test_binding_marshalling(L):
    """The binding's own checks, before anything reaches the library."""
    import torch
    cfg = L.make_config()
    t = torch.zeros(64, 4)
    with pytest.raises(ValueError, match="contiguous"):
        L.loco_compress(cfg, t.t(), 0x1000, 1, 0x2000, 0x3000, stream=0)        # a transposed view
    with pytest.raises(ValueError, match="not supported"):
        L.loco_compress(cfg, torch.zeros(64, dtype=torch.float16), 0x1000, 1, 0x2000, 0x3000, stream=0)
    with pytest.raises(ValueError, match="same ranks"):
        L.loco_decode_reduce(cfg, [0x1000, 0x1100], [0x2000], 64, 0x3000, stream=0)
    # a non-OK status becomes LocoError carrying the status and the library's message
    with pytest.raises(L.LocoError) as ei:
        L.loco_decode_reduce(cfg, [0x1000] * 17, [0x2000] * 17, 64, 0x3000, stream=0)
    assert ei.value.status == L.LOCO_ERR_UNSUPPORTED and "LOCO_ERR_UNSUPPORTED" in str(ei.value)
    # dtype inference: bf16 and fp32 gradients map to the header's codes
    assert L._grad_dtype(torch.zeros(1, dtype=torch.bfloat16), None) == L.LOCO_BF16
    assert L._grad_dtype(torch.zeros(1), None) == L.LOCO_F32


def test_config_and_hparams_layout(L, tmp_path):
    """The ctypes mirrors of loco_config / loco_adam_hparams have the layout a C
    compiler gives the header's structs: every field's offset and both sizes."""
    import ctypes
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    structs = {"loco_config": L.loco_config, "loco_adam_hparams": L.loco_adam_hparams}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "loco.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = {}
    for line in subprocess.check_output([str(exe)], text=True).splitlines():
        cname, field, val = line.split()
        got[(cname, field)] = int(val)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)
    c = L.make_config(bits=8, block=128, beta=0.25, err_scale_mult=6.0, reset_period=512, fixed_scale=2.0 ** 19)
    assert (c.bits, c.block, c.scale_mode, c.fixed_scale, c.beta, c.err_scale_mult, c.reset_period) == \
        (8, 128, L.LOCO_SCALE_FIXED, 2.0 ** 19, 0.25, 6.0, 512)
