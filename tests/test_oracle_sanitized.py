"""The oracle's pins pass with the oracle built under AddressSanitizer and
UndefinedBehaviorSanitizer: no out-of-bounds access, use after free or
undefined arithmetic in the test infrastructure every parity claim rests on.

The sanitized library is built in a temporary directory and the pin suite
runs against it in a child process with the ASan runtime preloaded (the
Python interpreter itself is not instrumented).  Skipped where gcc has no
ASan runtime."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "wfst_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"),
        os.path.join(ROOT, "tests", "test_oracle_interval_prune.py")]

_CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import oracle
oracle._LIB_PATH = {lib!r}
oracle.build = lambda force=False: {lib!r}
import pytest
sys.exit(pytest.main([*{pins!r}, "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                      "-k", "not workloads_0_and_3"]))
"""


def _asan_runtime():
    try:
        p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True,
                           timeout=60).stdout.strip()
    except Exception:
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_pins_pass_under_address_and_undefined_behaviour_sanitizers():
    rt = _asan_runtime()
    if rt is None:
        pytest.skip("gcc has no AddressSanitizer runtime here")
    with tempfile.TemporaryDirectory() as tmp:
        lib = os.path.join(tmp, "liboracle.so")
        subprocess.run(["gcc", "-O1", "-g", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                        "-fno-omit-frame-pointer", "-o", lib, SRC, "-lm"],
                       check=True, capture_output=True)
        env = dict(os.environ, LD_PRELOAD=rt, ASAN_OPTIONS="detect_leaks=0",
                   UBSAN_OPTIONS="print_stacktrace=1")
        r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, lib=lib, pins=PINS)], cwd=ROOT,
                           env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout + r.stderr
    assert "AddressSanitizer" not in out and "runtime error" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
