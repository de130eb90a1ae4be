"""Build the CUDA library in-tree: paged_split_kv_03_gb300/_lib/libpda.so.

Every translation unit is compiled by nvcc for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked into
one shared library with the CUDA runtime linked statically, so the library
loads on a machine without a GPU (the runtime only looks for the driver on
the first CUDA call).
"""
from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libpda.so")

SOURCES = ["pda_plan.cpp", "pda_mma.cu", "pda_tc.cu", "pda_noalloc.cu", "pda_append.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpda.so")


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
            *ARCH, *extra]


STAMP = os.path.join(LIBDIR, "stamp")


def _stamp() -> str:
    """The host architecture plus a hash of every input of the build: a
    library built from other sources, or on another machine type, is stale."""
    h = hashlib.sha256(platform.machine().encode())
    paths = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    paths += [os.path.join(INCLUDE, "pda.h"), os.path.abspath(__file__)]
    for p in paths:
        if os.path.isfile(p):
            h.update(os.path.basename(p).encode())
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def _current() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _stamp()


def ptxas_reports():
    """{kernel (mangled name): (registers, stack bytes, spill store bytes,
    spill load bytes)} from the ptxas reports of the last build."""
    import re
    out = {}
    for f in sorted(os.listdir(LIBDIR)):
        if not (f.startswith("ptxas_") and f.endswith(".txt")):
            continue
        name = None
        for line in open(os.path.join(LIBDIR, f)):
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                name = m.group(1)
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, "
                          r"(\d+) bytes spill loads", line)
            if m and name:
                out[name] = [None, *(int(x) for x in m.groups())]
                continue
            m = re.search(r"Used (\d+) registers", line)
            if m and name in out and out[name][0] is None:
                out[name][0] = int(m.group(1))
    return {k: tuple(v) for k, v in out.items()}


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if stale) and return the path of libpda.so."""
    if not force and _current():
        return LIB
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        # ptxas's resource report (registers, stack, spills) of every kernel
        # is kept beside the library for the build checks
        extra = ["-Xptxas", "-v"] if src.endswith(".cu") else []
        cmd = [cc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if src.endswith(".cu"):
            with open(os.path.join(LIBDIR, "ptxas_" + os.path.splitext(src)[0] + ".txt"), "w") as f:
                f.write(r.stderr)
        return obj, r.stderr if ptxas_info else ""

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_stamp() + "\n")
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
