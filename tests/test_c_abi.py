"""libpf.so from a plain C program (tests/c/abi_decode.c): it compiles and links against the
library and the CUDA runtime on any machine, and on a GPU it runs the append, the decode and
the split through the C ABI and checks them against the oracle."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def build_c_program(out_dir) -> str:
    from paged_kv_decode_pf_gb300 import LIB_PATH, _build
    _build.build()
    cuda = _cuda_home()
    exe = os.path.join(str(out_dir), "abi_decode")
    cmd = ["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c", "abi_decode.c"),
           os.path.join(ROOT, "oracle", "pf_oracle.c"), os.path.join(ROOT, "workloads", "gen.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           "-L", os.path.dirname(LIB_PATH), "-l:" + os.path.basename(LIB_PATH),
           "-Wl,-rpath," + os.path.dirname(LIB_PATH),
           "-L", os.path.join(cuda, "lib64"), "-L", os.path.join(cuda, "targets", "sbsa-linux", "lib"),
           "-L", os.path.join(cuda, "targets", "x86_64-linux", "lib"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


def test_c_program_builds_and_links(tmp_path):
    assert os.path.exists(build_c_program(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_the_step(tmp_path):
    exe = build_c_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
