"""The oracle's pins under AddressSanitizer and UndefinedBehaviorSanitizer (the tinyllm page
runs its C code under ASan / UBSan): every oracle function the pins call -- attention with
sinks, scales and fp8 pools, split-KV, merges, slot mapping, scatter, gather, validation --
runs in an instrumented build, and any out-of-bounds access or undefined behaviour aborts the
run."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _asan_runtime():
    try:
        p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                           text=True, timeout=60).stdout.strip()
    except (OSError, subprocess.SubprocessError):
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_under_asan_and_ubsan():
    rt = _asan_runtime()
    if rt is None:
        pytest.skip("no ASan runtime for gcc on this machine")
    env = dict(os.environ, PA_ORACLE_SANITIZE="1", LD_PRELOAD=rt,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, out
    assert "ERROR: AddressSanitizer" not in out and "runtime error" not in out, out
