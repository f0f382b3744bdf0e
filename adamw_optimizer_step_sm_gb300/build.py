"""Builds the CUDA library in-tree: csrc/*.cu with nvcc for sm_103a and
csrc/*.cpp with g++, compiled in parallel and linked into
``_build/libadamw_sm.so`` (CUDA runtime linked statically)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libadamw_sm.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", f"-I{INCLUDE}", f"-I{CSRC}"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-Wall", "-Wextra",
             f"-I{INCLUDE}", f"-I{CSRC}",
             f"-I{os.path.join(CUDA_HOME, 'include')}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build adamw_sm")
    return cand


def _sources():
    cu = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, defines=(), out_dir: str | None = None) -> str:
    """Compile the library when a source is newer than it; returns its path.

    ``defines`` (NAME=VALUE strings) set the kernels' build-time tuning
    constants; such builds go to ``out_dir`` (load one with the environment
    variable ADAMW_SM_LIBRARY)."""
    build_dir = out_dir or BUILD_DIR
    lib_path = os.path.join(build_dir, LIB_NAME)
    if not force and not defines and out_dir is None and up_to_date():
        return LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp = _sources()
    dflags = [f"-D{d}" for d in defines]
    jobs = []
    objs = []
    for src in cu:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        jobs.append([nvcc, *NVCC_FLAGS, *dflags, "-Xptxas", "-v", "-c", src, "-o", obj])
        objs.append(obj)
    for src in cpp:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        jobs.append(["g++", *CXX_FLAGS, *dflags, "-c", src, "-o", obj])
        objs.append(obj)
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        logs = list(ex.map(_run, jobs))
    tmp = lib_path + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, lib_path)
    if verbose:
        for log in logs:
            sys.stdout.write(log)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    return lib_path


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser(description="build libadamw_sm.so for sm_103a")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--define", action="append", default=[], metavar="NAME=VALUE",
                    help="a build-time tuning constant, e.g. ADAMW_BULK=1")
    ap.add_argument("--out", default=None, help="output directory for a tuning build")
    a = ap.parse_args()
    print(build(force=a.force, verbose=True, defines=a.define, out_dir=a.out))
