"""The C-ABI layer's host code under AddressSanitizer and
UndefinedBehaviorSanitizer: libpstat.so is rebuilt with the host code
instrumented (device code unchanged), and the argument-check tests of
test_abi.py run against that build in a child process with the sanitizer
runtimes preloaded.  Any sanitizer report is fatal there, so the child fails
on the first out-of-bounds access, use after free, overflow or other
undefined behaviour in the argument checks, shard-plan construction and
workspace sizing.  Runs without a GPU."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    gcc = shutil.which("gcc")
    if not gcc:
        return None
    p = subprocess.run([gcc, f"-print-file-name={name}"], capture_output=True, text=True).stdout
    p = p.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_abi_checks_under_sanitizers():
    import torch

    if torch.cuda.is_available():
        pytest.skip("host-only check: the argument tests use made-up device pointers")
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not (asan and ubsan):
        pytest.skip("gcc sanitizer runtimes not found")
    from vocab_wide_token_gb300 import build

    try:
        lib = build.build_sanitized()
    except RuntimeError as e:
        pytest.skip(f"no CUDA toolchain for the sanitizer build: {e}")
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}", PSTAT_TEST_LIB=lib,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "AddressSanitizer" not in out and "runtime error" not in out, out[-4000:]
    assert " passed" in out
