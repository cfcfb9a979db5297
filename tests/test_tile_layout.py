"""The group layout of the tensor-core top-k (csrc/tile.h), checked on the
host: tests/tile_layout_check.cpp is compiled with g++ against the header and
run (CPU)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"


@pytest.mark.skipif(shutil.which("g++") is None or not os.path.isdir(CUDA_INC),
                    reason="needs g++ and the CUDA headers")
def test_group_layout_invariants():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "tile_layout_check")
        subprocess.run(["g++", "-O2", "-std=c++17",
                        "-I", os.path.join(ROOT, "dynamic_top_sparse_rank_b300", "csrc"),
                        "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC,
                        os.path.join(ROOT, "tests", "tile_layout_check.cpp"), "-o", exe],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-2000:]
