"""Builds libbq.so in-tree for GB300 (sm_103a) with nvcc.

    python -m block_quant_gb300.build [--force] [--verbose]

Translation units compile in parallel; the shared library links the CUDA
runtime statically and takes the driver entry points it needs at run time, so
loading it needs no GPU.  The output lives next to this file, in _lib/.
"""

import argparse
import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libbq.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
# per source: extra flags.  The step kernels must not contract fp32 mul+add into
# FMA (their results are reproduced bit for bit by the oracle).
SOURCES = {
    "api.cpp": [],
    "planner.cpp": [],
    "step_kernels.cu": ["-lineinfo", "-fmad=false"],
    "ns_gemm.cu": ["-lineinfo"],
}
HEADERS = ["bq_internal.h", "tmem_ptx.h"]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbq")


def _digest():
    h = hashlib.sha256()
    for name in sorted(list(SOURCES) + HEADERS):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "bq.h"), "rb") as f:
        h.update(f.read())
    h.update(repr((ARCH, COMMON, SOURCES)).encode())
    return h.hexdigest()


def build(force=False, verbose=False):
    """Compile (if sources changed) and return the path of libbq.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = os.path.join(OUT_DIR, "libbq.stamp")
    digest = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB
    cc = nvcc()
    objs = []
    cmds = []
    for name, extra in SOURCES.items():
        src = os.path.join(CSRC, name)
        obj = os.path.join(OUT_DIR, name + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *COMMON, *extra, "-c", src, "-o", obj])
    if verbose:
        cmds = [c[:1] + ["-Xptxas", "-v"] + c[1:] if c[-3].endswith(".cu") else c for c in cmds]

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        for cmd, r in ex.map(run, cmds):
            if r.returncode != 0 or verbose:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    tmp = LIB + ".tmp"
    link = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        print(" ".join(link))
        print(r.stdout + r.stderr)
        raise RuntimeError("link of libbq.so failed")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
