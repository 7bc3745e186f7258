"""Build of the CUDA library ``libssd.so`` (sm_103a only).

Each translation unit under ``csrc/`` is compiled by nvcc in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``; the objects are
linked into ``sampling_ssd_verify_gb300/libssd.so`` next to this file (the
CUDA runtime is linked statically, so the library has no runtime search-path
requirements).  No CMake, no torch extension machinery.
"""

from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libssd.so")
CHECKS_LIB_PATH = os.path.join(PKG, "libssd_checks.so")
SOURCES = ["ssd_stream_bf16.cu", "ssd_stream_f32.cu", "ssd_cache.cu", "ssd_api.cu",
           "ssd_noalloc.cu", "ssd_tree.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "ssd.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile and link libssd.so if it is missing or older than its sources.

    checks=True builds libssd_checks.so instead: every global, shared and
    workspace access of the kernels is bounds-checked (-DSSD_CHECKS); a failed
    check is recorded in the last 256 bytes of the workspace and the access is
    skipped.  It is a debugging aid, not the product path."""
    lib_path = CHECKS_LIB_PATH if checks else LIB_PATH
    out_dir = OUT_DIR + ("_checks" if checks else "")
    if not force and up_to_date(lib_path):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                    "-Xptxas", "-v" if verbose else "-O3"] + (["-DSSD_CHECKS"] if checks else [])
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT)))
    errors = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            errors.append(" ".join(cmd) + "\n" + out.decode(errors="replace"))
        elif verbose:
            print(out.decode(errors="replace"))
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs, check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
