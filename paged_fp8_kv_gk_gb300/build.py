"""Build the CUDA library (libgk.so) in-tree with nvcc for sm_103a.

Usage: ``python -m paged_fp8_kv_gk_gb300.build`` or ``build()`` from Python.
Translation units compile in parallel and link into one shared library with
the CUDA runtime linked statically, so loading it needs only the driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgk.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["gk_kernels.cu", "gk_api.cu", "gk_noalloc.cu", "gk_ingest.cu"]
HEADERS = ["gk_device.cuh", "gk_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cand, "bin", "nvcc")
    if os.path.exists(p):
        return p
    w = shutil.which("nvcc")
    if not w:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return w


def _stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [
        os.path.join(INCLUDE, h) for h in ("gk.h", "gk_testing.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, lib_path: str = LIB_PATH,
          defines: tuple = ()) -> str:
    """Compile every translation unit and link libgk.so (or, with `defines`,
    a variant at `lib_path`); returns the library's path."""
    if not force and not _stale(lib_path):
        return lib_path
    out_dir = os.path.dirname(lib_path)
    os.makedirs(out_dir, exist_ok=True)
    # objects go to a directory of this process's own, so that concurrent
    # builds (parallel test workers) never overwrite each other's files; the
    # library itself is replaced atomically
    objdir = os.path.join(out_dir, f"obj{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        log = obj + ".log"
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-I", INCLUDE, "-c",
               os.path.join(CSRC, src), "-o", obj]
        f = open(log, "w")
        procs.append((subprocess.Popen(cmd, stdout=f, stderr=subprocess.STDOUT), f, log, cmd))
        objs.append(obj)
    failed = []
    for p, f, log, cmd in procs:
        rc = p.wait()
        f.close()
        if rc != 0 or verbose:
            with open(log) as fh:
                text = fh.read()
            if rc != 0:
                failed.append(" ".join(cmd) + "\n" + text)
            elif verbose:
                sys.stderr.write(text)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
    os.replace(tmp, lib_path)
    for src in SOURCES:  # keep the ptxas reports (registers, spills) beside the library
        log = os.path.join(objdir, src.replace(".cu", ".o.log"))
        os.replace(log, os.path.join(out_dir, os.path.basename(log)))
    shutil.rmtree(objdir, ignore_errors=True)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
