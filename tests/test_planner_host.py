"""The attention planner on the host, without a GPU: tests/planner_check.cpp compiles the
library's host source (hw_api.cpp) with its kernel launchers stubbed out, builds thousands of
plans over random cache states, layouts and call kinds, and checks each against facts
computed from the tables alone (token coverage per KV head, pieces inside pages and tiles,
rotation table from the layouts' view definitions, causal cuts and output rows, the fused
append's token list, early-load flags)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime.h")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def test_planner_plans_cover_every_token_once(tmp_path):
    cxx = shutil.which("g++")
    cuda = _cuda_home()
    if not cxx or not cuda:
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "planner_check")
    lib = os.path.join(cuda, "lib64")
    if not os.path.isdir(lib):
        lib = os.path.join(cuda, "lib")
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", os.path.join(cuda, "include"),
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "shared_kv_concurrent_gb300", "csrc"),
                    os.path.join(HERE, "planner_check.cpp"), "-o", exe, "-L", lib, "-lcudart",
                    "-Wl,-rpath," + lib], check=True, capture_output=True, timeout=300)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "planner ok" in r.stdout
