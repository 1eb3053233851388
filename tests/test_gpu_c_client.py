"""The C ABI from a plain C program: tests/c_client/sdpa_client.c links
libsdpa.so and the C oracle, allocates with the CUDA runtime, calls
sdpa_forward (device buffers) and sdpa_forward_host (page-locked host
buffers), and checks every output row against the oracle (2e-2 of the
row's scale).  No Python or torch is on that path."""
import os
import shutil
import subprocess

import pytest

import oracle
import transformer_scaled_dot_02_gb300 as sd
from transformer_scaled_dot_02_gb300 import build as sd_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_root():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_client(tmp_path):
    sd_build.build()
    lib_dir = os.path.dirname(sd.LIB_PATH)
    oracle_dir = os.path.dirname(oracle.build())
    cuda = _cuda_root()
    exe = str(tmp_path / "sdpa_client")
    cmd = ["gcc", "-std=c11", "-O2", os.path.join(HERE, "c_client", "sdpa_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", lib_dir, "-l:libsdpa.so", "-Wl,-rpath," + lib_dir,
           "-L", oracle_dir, "-l:liboracle.so", "-Wl,-rpath," + oracle_dir,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"),
           "-lm", "-o", exe]
    subprocess.check_call(cmd)
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "c client ok" in run.stdout
