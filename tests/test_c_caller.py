"""libbsmooth from a plain C program: the header compiles as C11 on its own
(no CUDA header), the library links, and a GPU run smooths worked example A."""
import os
import shutil
import subprocess

import pytest

import blocked_floyd_warshall_gb300 as bsm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_caller.c")
LIBDIR = os.path.dirname(bsm.LIBRARY_PATH)


def compile_caller(tmp_path, with_cuda):
    exe = tmp_path / ("caller_cuda" if with_cuda else "caller")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I" + os.path.join(ROOT, "include"),
           SRC, "-L" + LIBDIR, "-lbsmooth", "-Wl,-rpath," + LIBDIR, "-o", str(exe)]
    if with_cuda:
        cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
        cmd[1:1] = ["-DWITH_CUDA", "-I" + os.path.join(cuda, "include")]
        cmd += ["-L" + os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    link = os.path.join(LIBDIR, "libbsmooth.so")
    assert os.path.exists(link)
    subprocess.run(cmd, check=True)
    return exe


@pytest.fixture(scope="module")
def built():
    if shutil.which("gcc") is None:
        pytest.skip("gcc unavailable")
    bsm.build()


def test_c_caller_host_checks(built, tmp_path):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("host-only run is for GPU-less hosts; the GPU test covers it")
    except ImportError:
        pass
    exe = compile_caller(tmp_path, with_cuda=False)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr


@pytest.mark.gpu
def test_c_caller_gpu(built, tmp_path):
    exe = compile_caller(tmp_path, with_cuda=True)
    out = subprocess.run([str(exe), "gpu"], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "abi_caller: ok" in out.stdout
