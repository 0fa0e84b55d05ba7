"""The C ABI from a plain C11 program (tests/c_caller/caller.c): the header
compiles as C, the program links against liblayerattn.so, its argument
checks run without a device (CPU), and on a GPU its bf16 and fp32 calls
match the oracle's C entry point."""
import os
import shutil
import subprocess

import pytest

import oracle
from layer_attn_fwd_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "caller.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    build.build()
    oracle.build()
    exe = str(tmp_path / "caller")
    lib_dir = os.path.dirname(build.LIB)
    orc_dir = os.path.dirname(oracle.build())
    cuda_lib = os.path.join(CUDA, "lib64")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SRC, "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-llayerattn", "-L", orc_dir, "-loracle", "-L", cuda_lib, "-lcudart", "-lm",
           f"-Wl,-rpath,{lib_dir}:{orc_dir}:{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_caller_builds_and_validates_arguments(tmp_path):
    exe = _compile(tmp_path)
    r = subprocess.run([exe, "--abi"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "abi checks ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_caller_on_the_gpu(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe = _compile(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "C caller ok" in r.stdout, r.stdout + r.stderr
