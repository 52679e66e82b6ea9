"""The C ABI from plain C: tests/c_abi/abi_check.c includes include/lce.h and
include/lce_testing.h as C99, links liblce.so with gcc and runs its
host-side checks (no GPU, no Python, no torch in the client)."""

import os
import shutil
import subprocess

import pytest

from linear_cross_entropy_lce_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "linear_cross_entropy_lce_gb300")


def test_c99_client_builds_links_and_runs(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    _build.build()
    exe = str(tmp_path / "abi_check")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-L", PKG, "-llce", f"-Wl,-rpath,{PKG}",
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "C-ABI-OK" in r.stdout, r.stdout + r.stderr
