"""Builds libattn.so in-tree with nvcc for sm_103a.

The CUDA translation units compile in parallel and link into
attention_fwd_bwd_gb300/_lib/libattn.so. A content hash of the sources and
flags is stored next to the library, so an unchanged tree is not rebuilt.
"""
import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libattn.so")
# The bounds-checked build (-DATTN_DEBUG_BOUNDS): the same kernels with index
# checks that record ATTN_ERR_BOUNDS and skip the access; for tests only.
LIB_DEBUG = os.path.join(LIBDIR, "libattn_debug.so")
SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_bwd.cu", "attn_bwd_dvec.cu", "attn_noalloc.cu", "attn_sparse.cu",
           "attn_sparse_bwd.cu"]
HEADERS = ["attn_common.cuh", "attn_items.cuh", "attn_sparse.cuh", "sm100_ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _digest(extra=()):
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "attn.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force=False, verbose=False, debug=False):
    """Compile libattn.so (debug=True: libattn_debug.so, the bounds-checked
    build) if missing or stale; returns its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    lib = LIB_DEBUG if debug else LIB
    extra = ["-DATTN_DEBUG_BOUNDS"] if debug else []
    stamp = os.path.join(LIBDIR, "libattn_debug.sha256" if debug else "libattn.sha256")
    digest = _digest(extra)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib
    nvcc = _nvcc()
    objdir = os.path.join(LIBDIR, "obj_debug" if debug else "obj")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc] + ARCH + FLAGS + extra + ["-I", os.path.join(ROOT, "include"), "-c",
                                               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
