"""The forward's CUDA-core kernels checked on the CPU under host emulation
(tests/emu). They compile from the library's own kernel files with g++, and
every GPU thread is a fiber on the host:
- the row-wise exact top-k, the gather and window attention (plain and
  grouped heads) and the boundary smoothing, against the fp64 oracle: top-k
  bit for bit, attention within the GPU tests' tolerances;
- the selection stages of the tensor-core top-k (the bound from the group
  maxima, the candidate sort), fed group maxima and candidate lists built
  from exact scores. Their answers match bit for bit, and rows overflow
  exactly as they should.
A second build of each under AddressSanitizer runs a smaller set, so an
access outside any buffer fails the test. All run in child processes.

The tensor-core kernels (the score passes, the window band tiles, the
projection) use tcgen05, TMA and mbarriers, which have no host stand-in. The
GPU parity tests cover them."""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CHECK = os.path.join(HERE, "emu", "fwd_check.py")
TILE_CHECK = os.path.join(HERE, "emu", "tile_check.py")
sys.path.insert(0, os.path.join(HERE, "emu"))
import fwd_check  # noqa: E402
import tile_check  # noqa: E402

needs_gxx = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")


def _run(lib, *args, env=None, check=CHECK):
    r = subprocess.run([sys.executable, check, lib, *args], capture_output=True, text=True,
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


@needs_gxx
def test_tile_selection_stages_under_emulation(tmp_path):
    rc, out = _run(tile_check.build(str(tmp_path)), check=TILE_CHECK)
    assert rc == 0, out[-3000:]


@needs_gxx
@pytest.mark.skipif(_asan_runtime() is None, reason="needs the AddressSanitizer runtime")
def test_tile_selection_stages_stay_in_bounds_under_asan(tmp_path):
    lib = tile_check.build(str(tmp_path), asan=True)
    env = dict(os.environ, LD_PRELOAD=_asan_runtime(), ASAN_OPTIONS="detect_leaks=0")
    rc, out = _run(lib, "small", env=env, check=TILE_CHECK)
    assert rc == 0 and "ERROR: AddressSanitizer" not in out, out[-3000:]
