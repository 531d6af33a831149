"""The boundary is a C ABI: include/pa.h compiles as strict C99 (-pedantic,
warnings as errors) and a C program linked against libpa_gb300.so drives
the host-side entry points (tests/c_abi_check.c: version and status
strings, the block manager through fork, copy on write, stats and swap, and
a host-side argument rejection).  CPU only: nothing it calls touches a GPU."""

import os
import shutil
import subprocess

import pytest

from paged_kv_cache_124_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c99_client_builds_and_runs():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(api.library_path())
    out_dir = os.path.join(ROOT, "_build", "c_abi")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "c_abi_check")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_check.c"), "-L", lib_dir, "-lpa_gb300", "-Wl,-rpath," + lib_dir,
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
