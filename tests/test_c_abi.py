"""The C ABI used from C: tests/c/abi_smoke.c links libloco.so and libcudart
directly (no Python binding), allocates its own device buffers and checks the
hand-derived worked example bit for bit."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "bit_gradient_compression_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    from bit_gradient_compression_gb300 import build
    build.build()
    out = str(tmp_path_factory.mktemp("cabi") / "abi_smoke")
    libdirs = [os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"),
               os.path.join(CUDA, "targets", "sbsa-linux", "lib"), os.path.join(CUDA, "targets", "x86_64-linux", "lib")]
    ldflags = []
    for d in libdirs:
        if os.path.isdir(d):
            ldflags += ["-L", d, f"-Wl,-rpath,{d}"]
    subprocess.check_call(["gcc", "-std=c11", "-O1", "-Wall", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c", "abi_smoke.c"), "-o", out,
                           "-L", PKG, f"-Wl,-rpath,{PKG}", "-lloco", *ldflags, "-lcudart"])
    return out


def test_c_abi_cpu(exe):
    r = subprocess.run([exe, "cpu"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_abi_gpu(exe):
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
