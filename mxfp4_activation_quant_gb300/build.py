"""Build librmsq.so (the CUDA kernels and the C ABI) for sm_103a with nvcc.

The translation units compile in parallel, then link into one shared
library under ``_build/``. No fast-math: denormals are kept, and division
and square root stay IEEE, as the kernels' bit-exactness needs.

``build(debug=True)`` makes ``librmsq_debug.so`` with RMSQ_DEBUG defined: an
index check before every global store of the kernels (a failed check is
reported by rmsq_sync_status as RMSQ_ERR_BOUNDS). The binding loads it when
the environment sets RMSQ_DEBUG=1; it exists for the tests.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "librmsq.so")
DEBUG_LIB = os.path.join(OUT_DIR, "librmsq_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-I", INCLUDE]


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "rmsq.h"))
    return files


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    obj_dir = os.path.join(OUT_DIR, "debug") if debug else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= max(os.path.getmtime(p) for p in _deps())):
        return lib
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DRMSQ_DEBUG"] if debug else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
