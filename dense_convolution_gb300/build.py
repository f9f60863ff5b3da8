"""Build the CUDA library in-tree: one nvcc process per translation unit (in
parallel), then one shared-object link.  Output:
``dense_convolution_gb300/libconv2d_gb300.so`` (git-ignored).

Only sm_103a code is generated (``-gencode arch=compute_103a,code=sm_103a``);
nvcc cross-compiles it without a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libconv2d_gb300.so")
SOURCES = ["api.cu", "transforms.cu", "conv_fp32.cu", "conv_tc.cu", "winograd.cu", "static_workspace.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-I", os.path.join(ROOT, "include"), *extra]


def _deps_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "conv2d.h"),
                                                                  os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; skip when the library is newer than every source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        out = os.path.join(OBJ, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", out]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, out, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose or r.returncode != 0 or ptxas_info:
            sys.stderr.write(f"--- {s}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(s for s, _ in failed))
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc, "-shared", *ARCH, "-o", tmp, *[o for _, o, _ in results]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
