"""The C ABI from plain C: tests/c/abi_example.c includes only include/ep.h and the CUDA
runtime's header and links libep_gb300.so.  On the CPU it must compile and link as C11 (the
header is valid C); on a GPU it must run and match its hand-derived values."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")
LIBDIR = os.path.join(ROOT, "combine_topk_ids_histogram_gb300", "_build")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA runtime headers are not available")
    if not os.path.exists(os.path.join(LIBDIR, "libep_gb300.so")):
        pytest.skip("libep_gb300.so is not built")
    exe = str(tmp_path / "abi_example")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", LIBDIR, "-lep_gb300",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{LIBDIR}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    _build(tmp_path)


@pytest.mark.gpu
def test_c_caller_runs(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI example ok" in r.stdout
