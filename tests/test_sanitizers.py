"""Host sanitizers: the CPU oracle and the C ABI's host-side argument
validation run under AddressSanitizer and UndefinedBehaviorSanitizer.

Each test builds the sanitized variant (KVQ_SANITIZE=1: the oracle with gcc
-fsanitize=address,undefined; the library's host code through nvcc with the
same flags, its device code as PTX only, since nothing here launches a kernel)
and re-runs an existing CPU test module in a child process with the ASan
runtime preloaded.  Any sanitizer report aborts the child (leak detection is
off: the Python interpreter itself is not instrumented).  No GPU is needed.
"""
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT


def _runtime(name):
    r = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True)
    path = r.stdout.strip()
    return path if r.returncode == 0 and os.path.isabs(path) and os.path.exists(path) else None


def _run_under_sanitizers(test_file):
    asan = _runtime("libasan.so")
    if asan is None:
        pytest.skip("no AddressSanitizer runtime for this gcc")
    env = dict(os.environ, KVQ_SANITIZE="1", LD_PRELOAD=asan,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1:halt_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "not gpu", "-p", "no:cacheprovider",
                        os.path.join("tests", test_file)], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    out = r.stdout + r.stderr
    assert "ERROR: AddressSanitizer" not in out and "runtime error:" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
    return out


def test_oracle_under_asan_and_ubsan():
    """Every oracle pin (store, fp16 / e4m3 conversions, attention, split-T,
    prefill, TQ4, gather) with the sanitized oracle."""
    out = _run_under_sanitizers("test_oracle_pins.py")
    assert " passed" in out


def test_abi_validation_under_asan_and_ubsan():
    """The C ABI's host-side checks (every entry point's rejections, the
    workspace geometry, the no-allocation entry's ordering) with the sanitized
    library."""
    from bit_quantized_kv_store_gb300 import build   # noqa: F401  (the child builds its own variant)
    out = _run_under_sanitizers("test_abi.py")
    assert " passed" in out
