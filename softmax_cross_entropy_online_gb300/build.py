"""Build the library in-tree: nvcc for sm_103a, one process per translation unit.

Produces ``_lib/libce_gb300.so`` next to this file.  The CUDA runtime is
linked statically, so the library needs only the driver at run time.
"""

from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libce_gb300.so")
HASH_PATH = os.path.join(OUT_DIR, "build.hash")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _sources():
    units = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    headers = sorted(f for f in os.listdir(CSRC) if f.endswith(".cuh"))
    return units, headers


def _digest(units, headers) -> str:
    h = hashlib.sha256()
    h.update(" ".join(NVCC_FLAGS).encode())
    for f in units + headers:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(ROOT, "include", "ce_gb300.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ and link the shared library; returns its path."""
    units, headers = _sources()
    digest = _digest(units, headers)
    if not force and os.path.exists(LIB_PATH) and os.path.exists(HASH_PATH):
        with open(HASH_PATH) as fh:
            if fh.read().strip() == digest:
                return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for u in units:
        obj = os.path.join(OUT_DIR, u[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, u), "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        procs.append((u, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for u, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(u)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        sys.stderr.write(r.stdout.decode(errors="replace"))
        raise RuntimeError("linking libce_gb300.so failed")
    os.replace(tmp, LIB_PATH)
    with open(HASH_PATH, "w") as fh:
        fh.write(digest + "\n")
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
