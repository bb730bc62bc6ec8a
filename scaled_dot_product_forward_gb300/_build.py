"""Compile the sm_103a shared library in place (nvcc, no cmake).

``build()`` writes ``libsdpa_gb300.so`` next to this file.  Each translation
unit is compiled by its own nvcc process, in parallel, for exactly one target:
``-gencode arch=compute_103a,code=sm_103a``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB_NAME = "libsdpa_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["sdpa_fwd_sm103a.cu", "sdpa_fwd64_sm103a.cu", "sdpa_sparse_sm103a.cu", "sdpa_api.cpp"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the sm_103a library cannot be built")
    return cand


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "sdpa.h"))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build ``libsdpa_gb300.so`` if any source is newer; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    with tempfile.TemporaryDirectory(prefix="sdpa_build_") as tmp:
        procs, objs = [], []
        for src in SOURCES:
            obj = os.path.join(tmp, os.path.splitext(src)[0] + ".o")
            cmd = [nvcc, *GENCODE, *COMMON, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                print(" ".join(cmd))
            procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                           stderr=subprocess.STDOUT), cmd))
            objs.append(obj)
        for p, cmd in procs:
            out, _ = p.communicate()
            if p.returncode != 0:
                raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{out.decode()}")
        tmp_lib = os.path.join(tmp, LIB_NAME)
        link = [nvcc, *GENCODE, "-shared", "-o", tmp_lib, *objs]
        r = subprocess.run(link, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
        shutil.copyfile(tmp_lib, LIB_PATH + ".tmp")
        os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
