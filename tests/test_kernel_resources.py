"""Compile-time resource checks of the kernels (no GPU needed).

Each translation unit is compiled for sm_103a with the library's own flags
plus -Xptxas -v, and the assembler's per-kernel report is checked: no kernel
spills registers or uses a stack frame, and the kernels whose measured
occupancy depends on their register count stay within it (the int8-error
sender and Adam within their launch bounds of 3 CTAs of 256 threads per SM,
85 registers; the warp-local 4-bit decode within its 4 or 3 CTAs per SM).
"""
import concurrent.futures as cf
import os
import re
import shutil
import subprocess

import pytest

from bit_gradient_compression_gb300 import build as B

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")

ENTRY = re.compile(r"Compiling entry function '([^']+)'")
STACK = re.compile(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads")
REGS = re.compile(r"Used (\d+) registers")


@pytest.fixture(scope="module")
def report(tmp_path_factory):
    """{mangled kernel name: (registers, stack bytes, spill store bytes, spill load bytes)}"""
    out_dir = tmp_path_factory.mktemp("ptxas")

    def one(src):
        cmd = [B.nvcc(), *B.NVCC_FLAGS, "-Xptxas", "-v", "-c", os.path.join(B.CSRC, src),
               "-o", os.path.join(str(out_dir), src + ".o")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        return r.stderr

    with cf.ThreadPoolExecutor(len(B.SOURCES)) as ex:
        logs = list(ex.map(one, B.SOURCES))
    kernels, cur = {}, None
    for log in logs:
        for line in log.splitlines():
            m = ENTRY.search(line)
            if m:
                cur = m.group(1)
                kernels[cur] = [None, None, None, None]
                continue
            if cur is None:
                continue
            m = STACK.search(line)
            if m:
                kernels[cur][1:] = [int(m.group(1)), int(m.group(2)), int(m.group(3))]
            m = REGS.search(line)
            if m:
                kernels[cur][0] = int(m.group(1))
    assert kernels, "no kernel report parsed"
    return {k: tuple(v) for k, v in kernels.items()}


def test_every_kernel_reported(report):
    for family in ("k_compress", "k_decode_reduce", "k_adam", "k_sgd"):
        assert any(family in k for k in report), family
    assert all(None not in v for v in report.values())


def test_no_spills_no_stack(report):
    bad = {k: v for k, v in report.items() if v[1] or v[2] or v[3]}
    assert not bad, bad


def test_register_budgets(report):
    # the int8-error sender: k_compress_staged<bits, block, bf16, E8 = true, fixed, EL, S>,
    # 2 code widths x 3 blocks x 2 gradient types x 2 scale modes, within its launch bound
    # of 3 CTAs per SM (85 registers)
    e8 = [(k, v[0]) for k, v in report.items() if re.search(r"k_compress_stagedILi\dELi\d+ELb[01]ELb1E", k)]
    assert len(e8) == 24 and all(r <= 85 for _, r in e8), e8
    adam = [(k, v[0]) for k, v in report.items() if "k_adam" in k]
    assert adam and all(r <= 85 for _, r in adam), [a for a in adam if a[1] > 85]
    # the warp-local 4-bit decode k_decode_reduce_wl<4, W, 16, group> is fitted for four
    # CTAs of 256 threads per SM at W = 1..6 (64 registers) and three at W = 7, 8 (85)
    wl = {(int(m.group(1)), int(m.group(2))): v[0] for k, v in report.items()
          if (m := re.search(r"k_decode_reduce_wlILi4ELi(\d+)ELi16ELi(\d+)E", k))}
    assert sorted({w for w, _ in wl}) == list(range(1, 17)), sorted(wl)
    assert all(r <= 64 for (w, _), r in wl.items() if w <= 6), wl
    assert all(r <= 85 for (w, _), r in wl.items() if w in (7, 8)), wl
