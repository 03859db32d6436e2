"""Builds libspecverify.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m speculative_decoding_block_verify_gb300.build [--force] [--verbose]

Each .cu file is compiled in parallel to an object, then the objects are linked into one
shared library (static CUDA runtime).  Output: speculative_decoding_block_verify_gb300/_build/.
"""

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libspecverify.so"
SOURCES = ["api.cu", "verify.cu", "markov_bias.cu", "pick_k.cu", "pipeline.cu", "walk.cu", "cost_curve.cu"]
HEADERS = ["common.cuh", "df.cuh", "draw.cuh", "host_util.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def lib_path():
    return os.path.join(OUT_DIR, LIB_NAME)


def _nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found (CUDA toolkit required to build the library)")
    return exe


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False, ptxas_verbose=False):
    """Compile (if stale) and return the path of libspecverify.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    include = os.path.join(ROOT, "include")
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(include, "specverify.h")]
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        if not force and not ptxas_verbose and not _stale(o, [s] + hdrs):
            return o, ""
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", include, "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return o, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    if verbose or ptxas_verbose:
        for (_, log), src in zip(results, SOURCES):
            if log:
                print(f"== {src}\n{log}", file=sys.stderr)
    lib = lib_path()
    if force or _stale(lib, objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print -Xptxas -v resource usage")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas))
