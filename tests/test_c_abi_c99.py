"""The header and the library from a C99 program (tests/abi_c99.c): the header compiles as
strict C99 with every warning an error, a C program links libnvfp4kv.so and resolves its
symbols, and the host-only calls (version, status strings, size and layout queries, argument
checks that fail before any CUDA call) return what the header promises."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "abi_c99.c")


@pytest.fixture(scope="module")
def lib_path():
    from nvfp4_paged_kv_gb300 import build
    return build.build()


def test_c99_program_builds_links_and_passes(lib_path, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_c99")
    libdir = os.path.dirname(lib_path)
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
           "-L", libdir, "-lnvfp4kv", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120,
                       env={k: v for k, v in os.environ.items() if k != "LD_PRELOAD"})
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("all checks passed"), r.stdout


def test_header_alone_is_a_complete_c_translation_unit(tmp_path):
    """Included first and alone, the header needs nothing from its includer."""
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    tu = tmp_path / "only_header.c"
    tu.write_text('#include "nvfp4_kv.h"\nint nvfp4kv_only_header(void) { return 0; }\n')
    for std in ("c99", "c11"):
        r = subprocess.run(["gcc", f"-std={std}", "-pedantic", "-Wall", "-Wextra", "-Werror",
                            "-I", os.path.join(ROOT, "include"), "-c", str(tu), "-o",
                            str(tmp_path / f"only_header_{std}.o")], capture_output=True,
                           text=True)
        assert r.returncode == 0, r.stderr


def test_host_calls_under_asan_and_ubsan(tmp_path):
    """The same C program linked against a copy of the library whose host code is instrumented
    with AddressSanitizer and UndefinedBehaviorSanitizer (the device code is unchanged): every
    host-only call and argument check runs with bounds, lifetime, overflow and shift checks, and
    any finding aborts the program."""
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from nvfp4_paged_kv_gb300 import build
    lib = build.build(sanitize=True)
    exe = str(tmp_path / "abi_c99_sanitized")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
           "-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
           "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
           "-L", libdir, "-lnvfp4kv", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = {k: v for k, v in os.environ.items() if k != "LD_PRELOAD"}
    env["ASAN_OPTIONS"] = "detect_leaks=0:protect_shadow_gap=0:abort_on_error=1"
    env["UBSAN_OPTIONS"] = "print_stacktrace=1:halt_on_error=1"
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("all checks passed"), r.stdout
