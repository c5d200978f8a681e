"""The C ABI from plain C: tests/c_abi/sgp_c_smoke.c is compiled with gcc against
include/sgp.h and the in-tree libsgp.so (plus the CUDA runtime for device memory), then run
as its own process: one small layer temporally and as a two-stage pipeline, both SGP_OK and
bit-identical, with no Python or PyTorch in the process."""
import os
import shutil
import subprocess

import pytest

from intra_spatial_pipelining_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _cuda_home() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_c_program_runs_temporal_and_pipelined_layer(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    assert os.path.exists(build.LIB), "libsgp.so is not built"
    cuda = _cuda_home()
    exe = str(tmp_path / "sgp_c_smoke")
    cmd = [gcc, "-std=c11", "-O2", "-Wall", "-I", build.INCLUDE, "-I", os.path.join(cuda, "include"),
           os.path.join(HERE, "c_abi", "sgp_c_smoke.c"), "-L", build.BUILD, "-lsgp",
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + build.BUILD, "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout
