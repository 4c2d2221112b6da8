"""Builds the C-ABI library ``_lib/libringattn.so`` in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library against the static CUDA runtime (the library loads
without a GPU or a driver; the runtime looks for the driver at the first CUDA
call). Usage: ``python -m sequence_exact_attention_gb300.build``.

A second, checked build ``_lib/libringattn_debug.so`` comes from the same
sources with ``-DRA_DEBUG_CHECKS``: there every global-memory access a kernel
computes from indices is tested against its tensor's extent, and a violation
sets ``RA_ERR_RANGE`` in the status word and skips the access. It exports the
same entry points; ``binding.use_library("debug")`` switches to it.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT, "libringattn.so")
LIB_DEBUG = os.path.join(OUT, "libringattn_debug.so")
VARIANTS = {"release": (LIB, OUT, []),
            "debug": (LIB_DEBUG, os.path.join(OUT, "debug"), ["-DRA_DEBUG_CHECKS"])}

SOURCES = ["plan.cpp", "api.cpp", "tensor_map.cpp", "merge.cu", "attn_simt.cu", "attn_tc.cu",
           "attn_bwd.cu", "bwd_noalloc.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
          "-I", os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            exe = cand
    if exe is None:
        raise RuntimeError("nvcc not found")
    return exe


def _compile(src, variant, verbose):
    _, objdir, defs = VARIANTS[variant]
    path = os.path.join(CSRC, src)
    obj = os.path.join(objdir, src + ".o")
    cmd = [nvcc(), *ARCH, *COMMON, *defs, "-c", path, "-o", obj]
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def _link(variant, objs):
    lib = VARIANTS[variant][0]
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


def build(verbose=False, jobs=None, variants=("release", "debug")):
    """Compile and link every variant (all translation units of all variants
    in one parallel pool); returns the path of the release library."""
    units = [(s, v) for v in variants for s in SOURCES]
    for v in variants:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
    jobs = jobs or min(len(units), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(lambda u: _compile(u[0], u[1], verbose), units))
    if verbose:
        for (_, log), (s, v) in zip(results, units):
            if log.strip() and v == "release":
                print(f"--- {s}\n{log}", file=sys.stderr)
    libs = {v: _link(v, [o for (o, _), (_, uv) in zip(results, units) if uv == v])
            for v in variants}
    return libs.get("release", LIB)


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
