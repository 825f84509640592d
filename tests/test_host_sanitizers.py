"""Host code under sanitizers (CPU).

The library's host code (argument checks, sizing arithmetic, status strings:
everything the C ABI runs before any GPU work) is built with
UndefinedBehaviorSanitizer, and the input generator (synth.c, the only other
C code) with AddressSanitizer and UndefinedBehaviorSanitizer.  A child
pytest runs the CPU tests that exercise them against those builds: the ABI
and budget tests, the generator's tests, and the oracle tests that draw their
inputs from the generator.  Any sanitizer report stops the child with an
error.  The GPU kernels have their own bounds-checked build
(test_gpu_checked.py)."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_host_code_under_sanitizers():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not asan or not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("no AddressSanitizer runtime")
    import __graft_entry__
    __graft_entry__._build_module().build(ubsan=True)
    env = dict(os.environ, FT_SANITIZE="1", SYNTH_SANITIZE="1", LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    tests = ["tests/test_abi.py", "tests/test_budget.py", "tests/test_synth.py", "tests/test_oracle_ffn.py",
             "tests/test_oracle_fp8.py", "tests/test_oracle_routing.py", "tests/test_oracle_cache.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *tests, "-m", "not gpu", "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "passed" in r.stdout
