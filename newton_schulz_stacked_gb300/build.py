"""Builds libmuonbank.so in-tree with nvcc for sm_103a.

Each .cu file compiles in parallel to an object under ``_build/``; the objects
link into ``newton_schulz_stacked_gb300/libmuonbank.so`` with the CUDA runtime
linked statically (the driver API is reached through the runtime's
entry-point query, so no libcuda link is needed).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import re
import shutil
import signal
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libmuonbank.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--diag-suppress", "177"]
# the compiler's NVVM stage (cicc) on the aarch64 hosts sometimes dies with a segmentation
# fault on the tensor-core source (about one compile in six to one in three, on the same
# inputs; not its stack: on x86 the file compiles within a 1 MiB stack); a file whose
# compiler crashed is compiled again on its own, up to this many attempts in all (all
# failing: ~5e-5 at 1 in 3).  Ordinary compile errors fail the build at once.
COMPILE_ATTEMPTS = 9
_DIAGNOSTIC = re.compile(r"\berror\b", re.IGNORECASE)


def _crashed(r) -> bool:
    """Whether a compile failed because a compiler process died on a signal (not on a diagnostic):
    nvcc itself killed by one, or nvcc reporting a stage that was, with no error message."""
    if r.returncode == 0:
        return False
    if r.returncode < 0 or r.returncode == 128 + signal.SIGSEGV:
        return True
    text = (r.stdout or "") + (r.stderr or "")
    return "Segmentation fault" in text and not _DIAGNOSTIC.search(text)


def _flags_stamp(extra_flags) -> str:
    """Hash of the compiler, architecture and flags a library is built with."""
    return hashlib.sha256("\0".join([*ARCH, *CFLAGS, *extra_flags]).encode()).hexdigest()


def _stamp_path() -> str:
    return LIB_PATH + ".flags"


def _up_to_date(extra_flags) -> bool:
    if not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < _deps_mtime():
        return False
    try:
        with open(_stamp_path()) as f:
            return f.read().strip() == _flags_stamp(extra_flags)
    except OSError:
        return False


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime():
    files = _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "muonbank.h"))
    return max(os.path.getmtime(f) for f in files)


def build_library(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link the library if a source is newer than it or it was built with other flags;
    returns its path."""
    extra_flags = list(extra_flags)
    if not force and _up_to_date(extra_flags):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    objs = [os.path.join(BUILD_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [nvcc, *ARCH, *CFLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    for i, (cmd, r) in enumerate(results):
        for _ in range(COMPILE_ATTEMPTS - 1):
            if not _crashed(r):
                break
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr + "retrying this file alone\n")
            cmd, r = compile_one((srcs[i], objs[i]))
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("link of libmuonbank.so failed")
    os.replace(tmp, LIB_PATH)
    with open(_stamp_path(), "w") as f:
        f.write(_flags_stamp(extra_flags) + "\n")
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
