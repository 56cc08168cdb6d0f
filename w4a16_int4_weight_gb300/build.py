"""Build libw4a16.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the objects are linked into one
shared library with the CUDA runtime linked statically.  Rebuilds only when a
source or header is newer than the library.

Also builds, where the Python headers are installed, the binding's CPython
marshalling module (csrc/py_fastcall.c -> _w4a16_fastcall); without them the
binding calls the library through ctypes alone.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import sysconfig

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libw4a16.so")
INCLUDE = os.path.join(ROOT, "include")
FASTCALL_SRC = os.path.join(CSRC, "py_fastcall.c")
FASTCALL = os.path.join(HERE, "_w4a16_fastcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libw4a16")
    return p


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _newest_input() -> float:
    files = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build_fastcall(force: bool = False) -> bool:
    """Compile the CPython marshalling module if the Python headers exist."""
    if not force and os.path.exists(FASTCALL) and os.path.getmtime(FASTCALL) >= os.path.getmtime(FASTCALL_SRC):
        return True
    inc = sysconfig.get_paths().get("include", "")
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc or not os.path.exists(os.path.join(inc, "Python.h")):
        return False
    tmp = FASTCALL + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-O2", "-shared", "-fPIC", "-I", inc, FASTCALL_SRC, "-o", tmp],
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("building the CPython marshalling module failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, FASTCALL)
    return True


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    build_fastcall(force)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"{src}:\n{text}")
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
