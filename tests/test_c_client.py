"""The C-ABI used from plain C: tests/c_abi_client.c includes only include/ep.h
and the CUDA runtime API, links the in-tree libep.so and checks its own results
(see that file). Here it is compiled and linked without a GPU; the gpu-marked
test builds and runs it."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_client.c")
PKG = os.path.join(ROOT, "combine_ep_route_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir: str) -> str:
    from combine_ep_route_gb300 import build
    build.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "c_abi_client")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe,
           "-L", PKG, "-lep", f"-Wl,-rpath,{PKG}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(str(tmp_path)))


@pytest.mark.gpu
def test_c_client_runs(tmp_path):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
