"""The per-device cache behind the library's launch set-up (kernel
attributes, register counts, SM counts, occupancy), checked on the host: the
header is plain C++, so tests/cpp/per_device_test.cpp compiles it with g++
and drives it with a fake in place of the CUDA queries (separate entries per
device, failures retried, out-of-range devices refused, one set-up under
concurrent callers)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_per_device_cache(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path / "per_device_test")
    subprocess.check_call([gxx, "-std=c++17", "-O1", "-pthread",
                           "-I", os.path.join(ROOT, "exact_attention_62_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "cpp", "per_device_test.cpp"), "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "per_device: ok" in r.stdout
