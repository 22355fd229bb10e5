"""Build the C-ABI shared library in-tree with nvcc for sm_103a (GB300)."""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "liblp_ragged.so"
SOURCES = ["lp_ragged.cu"]
HEADERS = ["lp_device.cuh", "lp_kernels.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def lib_path() -> str:
    return os.path.join(LIB_DIR, LIB_NAME)


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "lp_ragged.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    out = lib_path()
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, out: str | None = None,
          defines=()) -> str:
    """Compile the library if a source changed; return its path. ``defines`` (e.g.
    ``["LP_UNROLL=8"]``) override the kernel's tuning knobs; use with ``out``."""
    out = out or lib_path()
    if not force and not defines and out == lib_path() and up_to_date():
        return out
    os.makedirs(os.path.dirname(os.path.abspath(out)), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2",
           "-I", INCLUDE, "-I", CSRC, "-o", tmp]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [f"-D{d}" for d in defines]
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    if verbose or ptxas_verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
