"""The C ABI from plain C: tests/c_abi/plan_demo.c (C99, include/zs.h
only) is compiled with gcc against libzs.so and run.  Host calls only."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "zero_sharded_optimizer_bucket_gb300")


def test_plain_c_client(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    if not os.path.exists(os.path.join(PKG, "libzs.so")):
        pytest.skip("libzs.so not built")
    exe = str(tmp_path / "plan_demo")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror",
                    "-I" + os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "plan_demo.c"),
                    "-L" + PKG, "-lzs", "-Wl,-rpath," + PKG, "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("ok")
