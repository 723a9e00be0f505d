"""The C ABI from a C program: include/rd.h compiles as C, and a C caller
(tests/c_caller.c: CUDA runtime buffers, one grouped forward, a rejected call,
the status word, a direct host loop as the check) links against librd.so and
runs.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cc():
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("no CUDA headers")
    return cc


def test_header_compiles_as_c(tmp_path):
    cc = _cc()
    obj = str(tmp_path / "c_caller.o")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-c", SRC, "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), "-o", obj], check=True)
    assert os.path.getsize(obj) > 0


@pytest.mark.gpu
def test_c_caller_runs(tmp_path, rd_lib):
    cc = _cc()
    lib_dir = os.path.dirname(rd_lib.lib_path())
    exe = str(tmp_path / "c_caller")
    subprocess.run([cc, "-std=c11", SRC, "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA, "include"), "-L", lib_dir, "-lrd",
                    "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe],
                   check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c caller ok" in r.stdout, r.stdout + r.stderr
