"""The public header serves a plain C caller.

tests/c/abi_consumer.c sees nothing but include/muonbank.h: it is compiled as
strict C99 (warnings are errors), linked to libmuonbank.so, and run.  Its
checks use only the entry points that need no device (workspace sizes,
argument errors, status strings), so the test runs on any host.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c99_consumer_builds_and_runs(tmp_path):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("no C compiler")
    from newton_schulz_stacked_gb300.build import build_library
    libdir = os.path.dirname(build_library())
    exe = str(tmp_path / "abi_consumer")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c", "abi_consumer.c"), "-L", libdir, "-lmuonbank", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi consumer ok" in r.stdout
