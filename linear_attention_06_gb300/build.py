"""In-tree build of libkda.so (CUDA, sm_103a only).

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc for
``-gencode arch=compute_103a,code=sm_103a`` and linked into
``linear_attention_06_gb300/libkda.so``.  Objects go to ``_build/``.  No cmake.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkda.so")
HEADERS = [os.path.join(ROOT, "include", "kda.h")]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None, tag=None) -> str:
    """Compile (if stale) and return the path of libkda.so.

    With ``tag`` the objects and the library go to ``_build/<tag>/`` instead (a
    separately configured copy, e.g. a diagnostic build with extra ``-D`` flags);
    the package's own ``libkda.so`` is left alone."""
    obj_dir = os.path.join(BUILD, tag) if tag else BUILD
    lib = os.path.join(obj_dir, "libkda.so") if tag else LIB
    os.makedirs(obj_dir, exist_ok=True)
    deps_common = HEADERS + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    flags = CFLAGS + list(extra_flags or [])
    procs, objs = [], []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + deps_common):
            cmd = [NVCC] + ARCH + flags + ["-c", src, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"{s}\n{o}" for s, o in failed))
    if force or _stale(lib, objs):
        cmd = [NVCC] + ARCH + ["-shared", "-o", lib] + objs
        subprocess.run(cmd, check=True)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
