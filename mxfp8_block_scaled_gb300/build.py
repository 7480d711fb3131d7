"""Build the sm_103a shared library in-tree with nvcc (no torch extension
machinery, no cmake): each .cu file compiles in parallel, then one link.

    python -m mxfp8_block_scaled_gb300.build        # or build() from Python

Output: mxfp8_block_scaled_gb300/_lib/libmxfp8_gb300.so (git-ignored).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libmxfp8_gb300.so"
SOURCES = ("mx_abi.cu", "mx_quant.cu", "mx_gemm.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-Xptxas", "-v"] + ARCH
# MXFP8_DISPATCH_OVERRIDES=1 at build time: a measurement build whose GEMM
# dispatch reads MXFP8_GEMM_PAIR / _BN / _SPLIT / _SCHEDULE from the environment.
if os.environ.get("MXFP8_DISPATCH_OVERRIDES", "") == "1":
    NVCC_FLAGS.append("-DMXFP8_DISPATCH_OVERRIDES")


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False) -> str:
    """Compile every kernel for sm_103a and link the C-ABI library; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    out = lib_path()
    tmp = out + ".tmp"
    cmd = [nvcc(), "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
