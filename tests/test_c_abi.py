"""The C ABI from plain C: tests/c_abi/fa_c_smoke.c includes include/fa.h,
links libfa_gb300.so and the CUDA runtime (plus the oracle's C file, which
only this test program links), and calls fa_forward on its own device
buffers.  On the CPU the program must compile and link (the header is plain
C); on a GB300 it must run and match the oracle."""
import os
import shutil
import subprocess

import pytest

from tiled_online_softmax_attn_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "fa_c_smoke.c")
ORACLE_C = os.path.join(ROOT, "oracle", "oracle.c")


def cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def build_program(out_dir):
    lib = fa_build.build()
    libdir = os.path.dirname(lib)
    cuda = cuda_home()
    cuda_lib = os.path.join(cuda, "lib64")
    exe = os.path.join(out_dir, "fa_c_smoke")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), SRC, ORACLE_C, "-o", exe,
           "-L", libdir, "-l:" + os.path.basename(lib), "-L", cuda_lib, "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}:{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(build_program(str(tmp_path)))


@pytest.mark.gpu
def test_c_program_runs_and_matches_the_oracle(tmp_path):
    exe = build_program(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
