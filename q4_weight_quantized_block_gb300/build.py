"""Compile the CUDA / C++ sources in csrc/ into the in-tree libfak.so (sm_103a).

Every translation unit is compiled in parallel with nvcc (one -gencode,
sm_103a only), then linked into one shared library next to this file.  No
cmake, no torch extension machinery: the library has a plain C ABI
(include/fak.h) and is loaded with ctypes.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfak.so")

SOURCES = ["engine.cu", "batch.cu", "gemm.cu", "prefill.cu", "pack.cpp", "pack_device.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _needs(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    """Build libfak.so if any source or header is newer; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(INCLUDE, "fak.h")] + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                                  if f.endswith((".cuh", ".h"))]
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    objs, procs = [], []
    for s in srcs:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s + ".o")
        objs.append(obj)
        if force or _needs(obj, [src] + headers):
            cmd = [nvcc] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-ffp-contract=off",
                                   "-I" + INCLUDE, "-I" + CSRC, "-c", src, "-o", obj]
            if s.endswith(".cpp"):
                cmd = [nvcc, "-O3", "-std=c++17", "-x", "cu", "-Xcompiler", "-fPIC,-ffp-contract=off",
                       "-I" + INCLUDE, "-I" + CSRC, "-c", src, "-o", obj] + ARCH
            if verbose:
                print(" ".join(cmd))
            procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((s, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join("--- %s ---\n%s" % f for f in failed)
        raise RuntimeError("libfak build failed:\n" + msg)
    if force or _needs(LIB, objs):
        tmp = LIB + ".%d.tmp" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"]
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
