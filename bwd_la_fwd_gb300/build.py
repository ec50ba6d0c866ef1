"""Build the CUDA library in-tree: ``python -m bwd_la_fwd_gb300.build [--checked]``.

Every ``csrc/*.cu`` file is compiled for sm_103a only (``-gencode arch=compute_103a,code=sm_103a``) in
parallel, then linked into ``bwd_la_fwd_gb300/libla_gb300.so``.  No CMake, no torch extension
machinery: the library is a plain C-ABI shared object.

``checked=True`` builds the same sources with ``-DLA_CHECKED`` into ``libla_gb300_checked.so``: every
global-memory index that a kernel computes itself for a workspace array or the normaliser is checked
against the array's extent, and a violation is recorded as LA_ERR_BOUNDS in the workspace status word
instead of being performed.  It is a test build (the product loads ``libla_gb300.so``).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libla_gb300.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libla_gb300_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def _stale(obj: str, src: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    m = os.path.getmtime(obj)
    return any(os.path.getmtime(f) > m for f in [src, *deps])


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    nvcc = nvcc_path()
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    if checked:
        extra_flags = ("-DLA_CHECKED", *extra_flags)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(HERE, "..", "include", "*.h")))
    flags = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
             "--expt-relaxed-constexpr", *extra_flags]
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, src, deps):
            cmd = [nvcc, *flags, "-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    # relink whenever an object is newer than the library (also after a link that failed part-way)
    lib_stale = not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs)
    if force or procs or lib_stale:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-L" + cuda_lib_dir(nvcc), "-lcudart", "-ldl"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
