"""Compile the CUDA library in-tree for sm_103a (nvcc, no cmake)."""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "libfa_back.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh"))]
    out += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libfa_back.so next to this file; returns its path.  The translation units compile in
    parallel (one nvcc per file, objects in a temporary folder), then one link."""
    if not force and up_to_date():
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if verbose:
        flags.insert(0, "-Xptxas=-v")
    with tempfile.TemporaryDirectory(prefix="fa_back_build_") as obj_dir:
        jobs = []
        for src in sources():
            obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
            cmd = [nvcc(), *flags, "-c", src, "-o", obj]
            jobs.append((obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        failed = False
        for obj, proc in jobs:
            out, _ = proc.communicate()
            if proc.returncode != 0:
                failed = True
                sys.stderr.write(out)
            elif verbose:
                sys.stderr.write(out)
        if failed:
            raise RuntimeError("nvcc failed building libfa_back.so")
        r = subprocess.run([nvcc(), *ARCH, "-shared", *[o for o, _ in jobs], "-o", tmp], stdout=subprocess.PIPE,
                           stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout)
            raise RuntimeError("nvcc failed linking libfa_back.so")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
