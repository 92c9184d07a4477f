"""Build the sm_103a shared library libpa_gb300.so in-tree.

Each translation unit under csrc/ is compiled by nvcc in parallel, then the
objects are linked into ``paged_kv_cache_192_gb300/libpa_gb300.so`` (static
CUDA runtime, no torch dependency).  Objects are cached in ``_build/`` keyed
by a hash of the sources and flags, so an unchanged tree rebuilds in no time.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpa_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _digest(paths, extra) -> str:
    h = hashlib.sha1()
    for p in sorted(paths):
        with open(p, "rb") as f:
            h.update(p.encode() + b"\0" + f.read())
    h.update(" ".join(extra).encode())
    return h.hexdigest()[:16]


def _compile(src: str, obj: str, headers) -> str:
    if os.path.exists(obj):
        return obj
    tmp = obj + ".tmp.o"
    cmd = [nvcc()] + NVCC_FLAGS + ["-c", src, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, obj)
    return obj


def build(verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                     glob.glob(os.path.join(INCLUDE, "*.h")))
    hdr_digest = _digest(headers, NVCC_FLAGS)
    objs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = []
        for src in sources:
            key = _digest([src], [hdr_digest])
            obj = os.path.join(BUILD, f"{os.path.basename(src)}.{key}.o")
            objs.append(obj)
            futs.append(ex.submit(_compile, src, obj, headers))
        for f in futs:
            f.result()
    # objects of earlier sources or flags are not reused: drop them
    keep = {os.path.basename(o) for o in objs}
    for old in glob.glob(os.path.join(BUILD, "*.o")):
        if os.path.basename(old) not in keep:
            os.remove(old)
    link_key = _digest(objs, ["link"])
    stamp = os.path.join(BUILD, "lib.stamp")
    if os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == link_key:
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(link_key)
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
