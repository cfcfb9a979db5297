"""The backward kernels (csrc/attn_bwd.cu) checked on the CPU under host
emulation (tests/emu): the kernels and C entry points compiled with g++, every
GPU thread a fiber on the host, against the fp64 oracle. This checks their
indexing, lane layout and arithmetic before and besides the GPU parity tests.
A second build with AddressSanitizer runs a few cases so that any access
outside a buffer, workspace included, fails the test. Both run in a child
process, so a crash is a failure, not the end of the test session."""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CHECK = os.path.join(HERE, "emu", "bwd_check.py")
sys.path.insert(0, os.path.join(HERE, "emu"))
import bwd_check  # noqa: E402

needs_gxx = pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")


def _run(lib, *args, env=None):
    r = subprocess.run([sys.executable, CHECK, lib, *args], capture_output=True, text=True,
                       env=env, timeout=900)
    return r.returncode, r.stdout + r.stderr


@needs_gxx
def test_backward_kernels_match_the_oracle_under_emulation(tmp_path):
    rc, out = _run(bwd_check.build(str(tmp_path)))
    assert rc == 0, out[-3000:]


def _asan_runtime():
    try:
        r = subprocess.run(["g++", "-print-file-name=libasan.so"], capture_output=True, text=True)
    except OSError:
        return None
    p = r.stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


@needs_gxx
@pytest.mark.skipif(_asan_runtime() is None, reason="needs the AddressSanitizer runtime")
def test_backward_kernels_stay_in_bounds_under_asan(tmp_path):
    lib = bwd_check.build(str(tmp_path), asan=True)
    env = dict(os.environ, LD_PRELOAD=_asan_runtime(), ASAN_OPTIONS="detect_leaks=0")
    rc, out = _run(lib, "small", env=env)
    assert rc == 0 and "ERROR: AddressSanitizer" not in out, out[-3000:]
