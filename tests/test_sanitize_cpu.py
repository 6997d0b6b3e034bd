"""The oracle and the library's host code under AddressSanitizer and
UndefinedBehaviorSanitizer, on the CPU (no GPU calls).

* oracle/oracle.c with a C driver (tests/sanitize/oracle_driver.c) that calls
  every entry point on ordinary, empty and invalid arguments;
* the CUDA library built with sanitized host code (device code unchanged),
  loaded with the sanitizer runtimes preloaded, running the CPU tests of its
  host-side checks, size queries and planner.

Any sanitizer report fails the run (errors are not recoverable).
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True)
    path = p.stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


needs_gcc = pytest.mark.skipif(shutil.which("gcc") is None or _runtime("libasan.so") is None,
                               reason="gcc with the sanitizer runtimes is needed")


@needs_gcc
def test_oracle_under_sanitizers(tmp_path):
    exe = tmp_path / "oracle_driver"
    cmd = ["gcc", "-std=c11", "-O1", "-g", "-fsanitize=address,undefined",
           "-fno-omit-frame-pointer", "-fno-sanitize-recover=all", "-fopenmp", "-o", str(exe),
           os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
           os.path.join(ROOT, "oracle", "oracle.c"), "-lm"]
    subprocess.run(cmd, check=True)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1", OMP_NUM_THREADS="4")
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "Sanitizer" not in r.stderr and "runtime error" not in r.stderr, r.stderr


@needs_gcc
@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc is needed")
def test_library_host_code_under_sanitizers():
    from ggml_out_prod_gb300 import _build
    _build.build()                          # both builds current: nothing compiles below
    san = _build.build(sanitize=True)
    env = dict(os.environ, GGML_OUT_PROD_GB300_LIBRARY=san,
               LD_PRELOAD=" ".join([_runtime("libasan.so"), _runtime("libubsan.so")]),
               ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0")
    tests = [os.path.join(ROOT, "tests", f) for f in
             ("test_abi.py", "test_sizes_cpu.py", "test_plan_cpu.py")]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *tests], capture_output=True, text=True, timeout=600,
                       env=env, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "Sanitizer" not in r.stderr and "runtime error" not in r.stderr, r.stderr[-3000:]
