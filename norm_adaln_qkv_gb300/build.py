"""Build the C-ABI library ``libmh3_preattn.so`` in-tree with nvcc for sm_103a.

The translation units (the C ABI host code, kernel 1, the two forms of
kernel 2, the output projection, the MLP GEMMs, the e4m3 and NVFP4 kernels)
are compiled in parallel and linked with the CUDA runtime linked statically, so
the library loads on a machine without a GPU driver (the driver is resolved
on the first CUDA call).  Output: ``norm_adaln_qkv_gb300/libmh3_preattn.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmh3_preattn.so")
SOURCES = ["mh3_preattn.cu", "k1_norm_adaln.cu", "k2_qkv_gemm.cu", "k2_qkv_gemm_pair.cu",
           "out_proj.cu", "mlp.cu", "e4m3_quantize.cu",
           "k2_nvfp4_pair.cu", "nvfp4_quantize.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    for d in (CSRC, os.path.join(ROOT, "include")):
        for f in os.listdir(d):
            if os.path.getmtime(os.path.join(d, f)) > t:
                return True
    return os.path.getmtime(__file__) > t


def build(force: bool = False, verbose: bool = False, defines=(), out: str = LIB) -> str:
    """Compile and link the library if any source is newer; returns its path.

    ``defines`` (e.g. ``("MH3_GROUP_PAIRS=16",)``) are extra -D flags of a
    variant build, which goes to ``out`` (its objects beside it) instead of
    the package's own library."""
    if out == LIB and not defines and not force and not _stale():
        return LIB
    build_dir = BUILD if out == LIB else os.path.splitext(out)[0] + "_build"
    os.makedirs(build_dir, exist_ok=True)
    extra = [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, *_flags(extra)]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import argparse
    ap = argparse.ArgumentParser(description="build the CUDA library (or a variant of it)")
    ap.add_argument("-v", "--verbose", action="store_true", help="print ptxas resource usage")
    ap.add_argument("--define", action="append", default=[], help="extra -D flag (repeatable)")
    ap.add_argument("--out", default=LIB, help="library path of a variant build")
    a = ap.parse_args()
    print(build(force=True, verbose=a.verbose, defines=a.define, out=os.path.abspath(a.out)))
