"""The library build retries a compile whose compiler process crashed.

The compiler's NVVM stage on the aarch64 build hosts sometimes dies with a
segmentation fault on identical inputs; build_library retries such a file on
its own before it reports the failure.  The compiler is replaced here by a
fake that crashes a chosen number of times, so no nvcc runs.
"""
import os
import threading
import types

import pytest

from newton_schulz_stacked_gb300 import build as B


def _fake_compiler(crashes_for, calls):
    """subprocess stand-in: compiling `crashes_for`'s file fails that many times, then succeeds."""
    lock = threading.Lock()

    def run(cmd, capture_output=True, text=True):
        src = cmd[cmd.index("-c") + 1] if "-c" in cmd else None
        out = cmd[cmd.index("-o") + 1]
        with lock:
            calls.append(os.path.basename(src) if src else "link")
            n = calls.count(os.path.basename(src)) if src else 0
        name = os.path.basename(src) if src else None
        if name in crashes_for and n <= crashes_for[name]:
            return types.SimpleNamespace(returncode=139, stdout="", stderr="Segmentation fault\n")
        open(out, "wb").close()
        return types.SimpleNamespace(returncode=0, stdout="", stderr="")

    return types.SimpleNamespace(run=run)


@pytest.fixture
def sandbox(tmp_path, monkeypatch):
    monkeypatch.setattr(B, "BUILD_DIR", str(tmp_path / "objs"))
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libmuonbank.so"))
    monkeypatch.setattr(B, "_nvcc", lambda: "nvcc")
    return tmp_path


def test_crashed_compile_is_retried(sandbox, monkeypatch):
    calls = []
    monkeypatch.setattr(B, "subprocess", _fake_compiler({"mb_ns_gemm.cu": 2}, calls))
    path = B.build_library(force=True)
    assert os.path.exists(path)
    assert calls.count("mb_ns_gemm.cu") == 3            # two crashes, then the compile that succeeds
    assert calls.count("mb_api.cu") == 1 and calls.count("link") == 1


def test_a_file_that_always_crashes_fails_the_build(sandbox, monkeypatch):
    calls = []
    monkeypatch.setattr(B, "subprocess", _fake_compiler({"mb_ns_gemm.cu": 99}, calls))
    with pytest.raises(RuntimeError, match="mb_ns_gemm.cu"):
        B.build_library(force=True)
    assert calls.count("mb_ns_gemm.cu") == B.COMPILE_ATTEMPTS == 9   # the parallel attempt and eight retries
    assert "link" not in calls
    assert not os.path.exists(B.LIB_PATH)


def test_a_compile_error_fails_at_once(sandbox, monkeypatch):
    """An ordinary diagnostic is not a crash: the file is not compiled again."""
    calls = []

    def run(cmd, capture_output=True, text=True):
        src = cmd[cmd.index("-c") + 1] if "-c" in cmd else None
        calls.append(os.path.basename(src) if src else "link")
        if src and src.endswith("mb_api.cu"):
            return types.SimpleNamespace(returncode=2, stdout="", stderr='mb_api.cu(1): error: identifier "x" is undefined\n')
        open(cmd[cmd.index("-o") + 1], "wb").close()
        return types.SimpleNamespace(returncode=0, stdout="", stderr="")

    monkeypatch.setattr(B, "subprocess", types.SimpleNamespace(run=run))
    with pytest.raises(RuntimeError, match="mb_api.cu"):
        B.build_library(force=True)
    assert calls.count("mb_api.cu") == 1 and "link" not in calls


def test_a_library_built_with_other_flags_is_rebuilt(sandbox, monkeypatch):
    calls = []
    monkeypatch.setattr(B, "subprocess", _fake_compiler({}, calls))
    B.build_library(extra_flags=["-DPROBE=1"])
    n = calls.count("link")
    B.build_library(extra_flags=["-DPROBE=1"])          # same flags, sources unchanged: reused
    assert calls.count("link") == n
    B.build_library()                                   # other flags: built again
    assert calls.count("link") == n + 1
    B.build_library()
    assert calls.count("link") == n + 1
