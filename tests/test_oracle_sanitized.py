"""The oracle's pins, rerun against a build of the oracle's C source instrumented with
AddressSanitizer and UndefinedBehaviorSanitizer.

The pins check the oracle's values; this run also checks how it gets them: an out-of-bounds
read or write, a use after free, a signed overflow, a shift past the width or a misaligned
access anywhere on the paths the pins reach aborts the child process. The child is a plain
pytest run of the pin files with gcc's ASan runtime preloaded (a sanitized shared library
loaded through ctypes needs the runtime in the process before Python starts)."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_format.py", "tests/test_oracle_codec.py",
             "tests/test_oracle_attention.py", "tests/test_oracle_cold.py",
             "tests/test_oracle_scale_study.py"]


def _asan_runtime():
    try:
        out = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                             text=True, check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        return None
    return out if os.path.isabs(out) and os.path.exists(out) else None


@pytest.fixture(scope="module")
def sanitized_env():
    asan = _asan_runtime()
    if asan is None:
        pytest.skip("gcc has no AddressSanitizer runtime here")
    lib = oracle.build(sanitize=True)
    env = dict(os.environ, LD_PRELOAD=asan, NVFP4_ORACLE_LIB=lib,
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=1:detect_odr_violation=0",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    env.pop("PYTEST_ADDOPTS", None)
    return env, lib


def test_child_loads_the_sanitized_oracle(sanitized_env):
    env, lib = sanitized_env
    code = ("import oracle, numpy as np\n"
            "l = oracle._load()\n"
            "maps = open('/proc/self/maps').read()\n"
            "print(l._name)\n"
            "print('libasan' in maps, 'libubsan' in maps)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    name, flags = r.stdout.split("\n")[:2]
    assert name == lib
    assert flags == "True True"


def test_pins_pass_under_asan_and_ubsan(sanitized_env):
    env, _ = sanitized_env
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu", *PIN_FILES], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1200)
    tail = r.stdout[-3000:] + r.stderr[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
