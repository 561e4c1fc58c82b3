"""Build the sm_103a shared library ``_build/libsagefp4.so`` with nvcc.

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces the shared library.  The CUDA runtime is linked statically
and the driver API is reached through the runtime's entry-point query, so the
library loads (and its symbols resolve) on a machine without a GPU driver.

``build(debug_bounds=True)`` builds ``_build_debug/libsagefp4_debug.so``
instead: the same sources with SAGE_FP4_DEBUG_BOUNDS=1, in which the kernels
check every global-memory index they compute against its buffer, record a
failure as SAGE_FP4_EBOUNDS in the status word and skip that access.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsagefp4.so")
OUT_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(OUT_DEBUG, "libsagefp4_debug.so")
SOURCES = ["quant.cu", "attn.cu", "probe.cu", "api.cu", "noalloc.cu", "host_pipe.cu", "sagebwd.cu"]
HEADERS = ["ptx.cuh", "layout.cuh", "kernels.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "sage_fp4.h"))
    files.append(os.path.join(ROOT, "include", "sagebwd.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    out_dir, lib = (OUT_DEBUG, LIB_DEBUG) if debug_bounds else (OUT, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if debug_bounds:
        common += ["-DSAGE_FP4_DEBUG_BOUNDS=1"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
