"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer: every pin runs against a
copy of oracle.c built with -fsanitize=address,undefined (no recovery), in a child process
that preloads the ASan runtime.  A memory error or undefined behaviour in the oracle fails
the child."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import ctypes, sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
oracle._lib = oracle._bind(ctypes.CDLL({so!r}))
for pin in oracle_pins.ALL_PINS:
    pin()
print("pins", len(oracle_pins.ALL_PINS))
"""


def test_pins_under_asan_ubsan(tmp_path):
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("no ASan runtime for gcc here")
    so = tmp_path / "liboracle_san.so"
    src = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")
    subprocess.check_call(["gcc", "-O1", "-g", "-std=c11", "-fPIC", "-shared", "-fsanitize=address,undefined",
                           "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-o", str(so), src, "-lm"])
    env = dict(os.environ, LD_PRELOAD=asan, ASAN_OPTIONS="detect_leaks=0:abort_on_error=1",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, so=str(so))], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert "pins" in r.stdout
