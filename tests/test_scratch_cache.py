"""The static scratch array's address cache (csrc/scratch_cache.h) on the host, without a GPU.

csa_index_topk_static looks up the device address of its fixed scratch array once per device and context; a
lookup under another context (the device was reset and its context created again) must miss, so that a call never
launches a kernel with an address from a destroyed context.  The cache logic is plain C++ and is checked here by
compiling a small driver with g++ and running it.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_context_address_cache_invalidates_on_a_new_context(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "scratch_cache_check")
    src = os.path.join(ROOT, "tests", "scratch_cache_check.cpp")
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-pthread", src, "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
