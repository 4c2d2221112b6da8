"""Builds the C-ABI library ``_lib/libringattn.so`` in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library against the static CUDA runtime (the library loads
without a GPU or a driver; the runtime looks for the driver at the first CUDA
call). Usage: ``python -m sequence_exact_attention_gb300.build``.
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

SOURCES = ["plan.cpp", "api.cpp", "tensor_map.cpp", "merge.cu", "attn_simt.cu", "attn_tc.cu",
           "attn_bwd.cu"]

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


def _compile(src, verbose):
    path = os.path.join(CSRC, src)
    obj = os.path.join(OUT, src + ".o")
    cmd = [nvcc(), *ARCH, *COMMON, "-c", path, "-o", obj]
    if verbose and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def build(verbose=False, jobs=None):
    """Compile and link; returns the path of the shared library."""
    os.makedirs(OUT, exist_ok=True)
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for (o, log), s in zip(results, SOURCES):
            if log.strip():
                print(f"--- {s}\n{log}", file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
