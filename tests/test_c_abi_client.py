"""The C ABI used from plain C: tests/c_abi_client.c is compiled with gcc
against include/ar.h and libar_gb300.so (no Python, no C++ in the client)
and run, without a GPU for its argument checks and on the GPU for every
variant, reduce-scatter, all-gather and the host-buffer path, checked
against exact-integer closed forms."""
import os
import shutil
import subprocess

import pytest

from shot_allreduce_ranks_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if not shutil.which("gcc"):
        pytest.skip("gcc is not installed")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("CUDA headers not found")
    build.build()
    exe = str(tmp_path_factory.mktemp("c_client") / "c_abi_client")
    pkg = os.path.dirname(build.LIB)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "c_abi_client.c"),
           "-L", pkg, "-l:" + os.path.basename(build.LIB),
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + pkg, "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_argument_checks_without_gpu(client):
    r = subprocess.run([client, "--host-only"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failed" in r.stdout


@pytest.mark.gpu
def test_c_client_on_the_gpu(client):
    r = subprocess.run([client], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failed" in r.stdout
