"""Compile libspecverify.so in-tree for sm_103a with nvcc (no cmake)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libspecverify.so")
# the bounds-checked debug build: every checked row / chunk / token index that
# falls outside its extent is recorded in the status word (SPEC_ERR_DEVICE_BOUNDS)
LIB_CHECKED = os.path.join(LIBDIR, "libspecverify_checked.so")
SOURCES = ["spec_verify.cu", "round_driver.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".cpp"))]
    files.append(os.path.join(INCLUDE, "spec_verify.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _command(out: str, checked: bool, extra_flags=()):
    return ([nvcc_path(), "-O3", "-lineinfo", "-std=c++17", *ARCH, "-shared",
             "-Xcompiler", "-fPIC", "-cudart", "static", "-I", INCLUDE, "-I", CSRC]
            + (["-DSPEC_CHECK_BOUNDS"] if checked else []) + list(extra_flags)
            + ["-o", out] + [os.path.join(CSRC, s) for s in SOURCES])


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False,
          both: bool = False) -> str:
    """Build the shared library if any source is newer than it; return its path.
    checked=True builds the bounds-checked variant instead; both=True builds
    the two side by side (two nvcc processes) and returns the normal one."""
    targets = [(LIB_CHECKED if checked else LIB, checked)]
    if both:
        targets = [(LIB, False), (LIB_CHECKED, True)]
    todo = [(lib, chk) for lib, chk in targets if force or not up_to_date(lib)]
    if todo:
        os.makedirs(LIBDIR, exist_ok=True)
        procs = []
        for lib, chk in todo:
            cmd = _command(lib + ".tmp", chk, extra_flags)
            if verbose:
                print(" ".join(cmd))
            procs.append((lib, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
        for lib, pr in procs:
            out, err = pr.communicate()
            if pr.returncode != 0:
                raise RuntimeError(f"nvcc failed ({pr.returncode}) for {os.path.basename(lib)}:\n{out}\n{err}")
            if verbose and (out or err):
                print(out, err)
            os.replace(lib + ".tmp", lib)
    return targets[0][0]


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, both=True))
