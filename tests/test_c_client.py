"""The C ABI from plain C: tests/c_client/ep_c_client.c includes only
include/ep_layout.h and the CUDA runtime header, links the built library and
the CUDA runtime, and runs layout, dispatch and combine with device memory it
allocates itself.  Compiling it (with -Werror, as C99) runs anywhere; running
it needs a GPU."""
import os
import shutil
import subprocess

import pytest

from combine_ep_layout_03_gb300 import ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "ep_c_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def compile_client(out_dir) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(str(out_dir), "ep_c_client")
    libdir = os.path.dirname(ep.LIB_PATH)
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-ffp-contract=off",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-o", exe, ep.LIB_PATH, f"-Wl,-rpath,{libdir}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_and_client_compile_as_c99(tmp_path):
    compile_client(tmp_path)


@pytest.mark.gpu
def test_c_client_runs_the_path(tmp_path):
    exe = compile_client(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
