"""A C program runs a Muon step through the library, with device memory from the CUDA runtime.

tests/c/step_consumer.c uses include/muonbank.h and the CUDA runtime API only
(no Python, no PyTorch): it checks a zero-gradient slot against its exact
decay-only result and that two runs give the same bytes.
"""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _cuda_home():
    nvcc = shutil.which("nvcc")
    for cand in (os.environ.get("CUDA_HOME"), os.path.dirname(os.path.dirname(nvcc)) if nvcc else None,
                 "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    pytest.fail("CUDA toolkit headers not found")


def test_c_program_runs_a_step(tmp_path):
    gcc = shutil.which("gcc")
    assert gcc, "no C compiler"
    from newton_schulz_stacked_gb300.build import build_library
    libdir = os.path.dirname(build_library())
    cuda = _cuda_home()
    cudalib = os.path.join(cuda, "lib64")
    exe = str(tmp_path / "step_consumer")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-isystem", os.path.join(cuda, "include"), os.path.join(HERE, "c", "step_consumer.c"),
           "-L", libdir, "-lmuonbank", "-L", cudalib, "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudalib}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "step consumer ok" in r.stdout
