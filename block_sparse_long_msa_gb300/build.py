"""Build libmsa.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Every translation unit under csrc/ is compiled in parallel, then linked into
block_sparse_long_msa_gb300/_build/libmsa.so, and again with MSA_DEBUG_CHECKS into the checked
build _build/libmsa_debug.so (objects under _build/debug/).
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libmsa.so")
# the checked build: the same calls, with MSA_DEBUG_CHECKS (include/msa.h, "Checked build")
DEBUG_LIB = os.path.join(OUT, "libmsa_debug.so")
ROOT = os.path.dirname(HERE)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "--expt-relaxed-constexpr", "-DMSA_NVTX", "-I", os.path.join(ROOT, "include")]
VARIANTS = {LIB: (OUT, []), DEBUG_LIB: (os.path.join(OUT, "debug"), ["-DMSA_DEBUG_CHECKS"])}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose=False):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stdout + r.stderr)
    return r


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug: bool = True) -> str:
    """Compile libmsa.so (and, with debug, libmsa_debug.so); every translation unit of both
    libraries is compiled in one parallel pool.  Returns the path of libmsa.so."""
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                     + glob.glob(os.path.join(ROOT, "include", "*.h")))
    nvcc = _nvcc()
    libs = [LIB, DEBUG_LIB] if debug else [LIB]
    objs, jobs = {}, []
    for lib in libs:
        out_dir, defs = VARIANTS[lib]
        os.makedirs(out_dir, exist_ok=True)
        flags = NVCC_FLAGS + defs + (extra_flags or [])
        objs[lib] = []
        for src in sources:
            obj = os.path.join(out_dir, os.path.basename(src) + ".o")
            objs[lib].append(obj)
            if force or _stale(obj, [src] + headers + [__file__]):
                jobs.append([nvcc] + flags + ["-c", src, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda c: _run(c, verbose), jobs))
    for lib in libs:
        if force or jobs or _stale(lib, objs[lib]):
            tmp = lib + f".{os.getpid()}.tmp"
            _run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs[lib] +
                 ["-ldl"], verbose)
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
