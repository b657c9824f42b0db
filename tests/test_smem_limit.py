"""The launchers' (kernel, device) shared-memory limit table, on the CPU.

The routing, row-mover and one-launch dispatch kernels need more than the
default 48 KiB of dynamic shared memory, a limit raised per kernel and per
device. ``csrc/smem_limit.h`` keeps one record per (kernel, device) under a
lock, so one process may drive several GPUs. This builds a small host program
against that header with a fake raise function and runs it.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_smem_limit_table(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "smem_limit_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Wextra", "-Werror", "-pthread",
                    os.path.join(HERE, "smem_limit_check.cpp"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
