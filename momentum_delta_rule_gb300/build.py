"""Build ``libmdn.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each CUDA translation unit compiles in parallel to an object file under
``_build/``; the objects link into ``momentum_delta_rule_gb300/libmdn.so``.
No CMake, no torch extension machinery: the library exposes a plain C ABI
(``include/mdn.h``).
"""
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libmdn.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
NVCC = os.environ.get("NVCC", "nvcc")

COMMON = ["-O3", "-std=c++17", ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
          "-I" + INCLUDE, "-I" + CSRC]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths) if paths else 0.0


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link; returns the library path.  Raises on failure."""
    srcs = sources()
    os.makedirs(BUILD_DIR, exist_ok=True)
    hdr_t = max(_newest(headers()), os.path.getmtime(__file__))
    objs, procs = [], []
    for src in srcs:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) > max(os.path.getmtime(src), hdr_t)):
            continue
        cmd = [NVCC] + COMMON + list(extra_flags) + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), flush=True)
    if failed:
        msg = "\n".join("%s:\n%s" % f for f in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    if (force or procs or not os.path.exists(LIB_PATH)
            or os.path.getmtime(LIB_PATH) < _newest(objs)):
        tmp = LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = [NVCC, ARCH, "-shared", "-o", tmp] + objs + ["-lcublas"]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [])
