"""The split-KV work plan (host code) on random layouts: coverage, chunk
ranges, slot uniqueness and visual-cut alignment (tests/plan_check.cpp)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_mixed_precision_kvq_gb300", "csrc")


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda_runtime.h")):
            return c
    return None


def test_plan_invariants(tmp_path):
    cuda = _cuda_home()
    gxx = shutil.which("g++")
    if cuda is None or gxx is None:
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path / "plan_check")
    cmd = [gxx, "-O1", "-std=c++17", "-I" + os.path.join(ROOT, "include"), "-I" + CSRC,
           "-I" + os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "plan_check.cpp"),
           os.path.join(CSRC, "kvq_layout.cpp"), "-L" + os.path.join(cuda, "lib64"),
           "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True)
    r = subprocess.run([exe, "20000"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
    print(r.stdout.strip())
