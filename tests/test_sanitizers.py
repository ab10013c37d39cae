"""The host radix cache under AddressSanitizer and UndefinedBehaviorSanitizer
(a debug build of csrc/radix_cache.cpp with tests/native/cache_stress.cpp, a
randomised driver of every host call): no memory error, no undefined
behaviour, consistent counts, for several seeds.  Needs g++ with the
sanitizer runtimes; skipped where they are missing."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    cuda_inc = "/usr/local/cuda/include"
    exe = str(tmp_path / "cache_stress")
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fno-omit-frame-pointer",
           "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
           "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(ROOT, "radix_tree_prefix_gb300", "csrc"), "-I", cuda_inc,
           os.path.join(ROOT, "radix_tree_prefix_gb300", "csrc", "radix_cache.cpp"),
           os.path.join(ROOT, "tests", "native", "cache_stress.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        if "sanitize" in r.stderr and ("cannot find" in r.stderr or "not found" in r.stderr):
            pytest.skip("sanitizer runtimes missing")
        raise AssertionError(r.stderr[-3000:])
    return exe


def test_host_cache_under_sanitizers(tmp_path):
    exe = _build(tmp_path)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    for seed in (1, 2, 3, 4):
        r = subprocess.run([exe, str(seed), "6000"], capture_output=True, text=True, env=env,
                           timeout=600)
        out = r.stdout + r.stderr
        assert "AddressSanitizer" not in out and "runtime error" not in out, out[-4000:]
        assert r.returncode == 0, out[-4000:]
