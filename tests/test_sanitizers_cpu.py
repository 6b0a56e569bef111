"""The host side of the C ABI under AddressSanitizer and UndefinedBehaviorSanitizer.

libqsa_asan.so is the release library with api.cpp -- the argument checks
every call runs before anything reaches the device -- compiled by g++ with
-fsanitize=address,undefined (UB is fatal).  The CPU ABI tests then run in a
child process that loads it with the sanitizer runtimes preloaded: every
rejection path, the zero-token paths and the export checks execute under the
sanitizers, and any report fails the run.  No GPU is used.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    gxx = shutil.which("g++")
    if not gxx:
        pytest.skip("g++ not available")
    path = subprocess.run([gxx, f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(path) or not os.path.exists(path):
        pytest.skip(f"{name} not available")
    return path


def test_abi_checks_under_asan_and_ubsan():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    from sparse_selected_attention_gb300 import build
    lib = build.build_host_sanitized()
    # the library really carries the instrumentation
    syms = subprocess.run(["nm", "-D", "--undefined-only", lib], capture_output=True, text=True).stdout
    assert "__asan_report" in syms and "__ubsan_handle" in syms
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}", ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1", QSA_LIB=lib, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_abi_cpu.py"), "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert " passed" in r.stdout and "ERROR: AddressSanitizer" not in out and "runtime error" not in out
