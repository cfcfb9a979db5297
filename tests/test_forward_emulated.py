"""The forward's CUDA-core kernels checked on the CPU under host emulation
(tests/emu). The row-wise exact top-k, the gather and window attention (plain
and grouped heads) and the boundary smoothing are compiled from the library's
own kernel files with g++, every GPU thread a fiber on the host, and checked
against the fp64 oracle: top-k bit for bit, attention within the GPU tests'
tolerances. A second build under AddressSanitizer runs a smaller set, so an
access outside any buffer fails the test. Both run in a child process.

The tensor-core kernels (the tile scorer, the window band tiles, the
projection) use tcgen05, TMA and mbarriers, which have no host stand-in; the
GPU parity tests cover them."""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CHECK = os.path.join(HERE, "emu", "fwd_check.py")
sys.path.insert(0, os.path.join(HERE, "emu"))
import fwd_check  # noqa: E402

needs_gxx = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")


def _run(lib, *args, env=None):
    r = subprocess.run([sys.executable, CHECK, lib, *args], capture_output=True, text=True,
                       env=env, timeout=900)
    return r.returncode, r.stdout + r.stderr


def _asan_runtime():
    try:
        r = subprocess.run(["g++", "-print-file-name=libasan.so"], capture_output=True, text=True)
    except OSError:
        return None
    p = r.stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


@needs_gxx
def test_forward_kernels_match_the_oracle_under_emulation(tmp_path):
    rc, out = _run(fwd_check.build(str(tmp_path)))
    assert rc == 0, out[-3000:]


@needs_gxx
@pytest.mark.skipif(_asan_runtime() is None, reason="needs the AddressSanitizer runtime")
def test_forward_kernels_stay_in_bounds_under_asan(tmp_path):
    lib = fwd_check.build(str(tmp_path), asan=True)
    env = dict(os.environ, LD_PRELOAD=_asan_runtime(), ASAN_OPTIONS="detect_leaks=0")
    rc, out = _run(lib, "small", env=env)
    assert rc == 0 and "ERROR: AddressSanitizer" not in out, out[-3000:]
