"""Build libgbattn.so in-tree from csrc/*.cu for sm_103a (nvcc, parallel compiles).

Objects go to streaming_attention_flashattention_gb300/_build/, the shared library next
to this file.  The CUDA runtime is linked statically and the driver's tensor-map encoder
is looked up at run time, so the library loads on a machine without a GPU driver.

build(debug=True) builds the same sources with -DGBATTN_DEBUG_CHECKS into _build_debug/ and
libgbattn_debug.so: kernels that check the index of each global store against its buffer
and record a failed check in the device error word instead of writing (include/gbattn.h).
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgbattn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libgbattn_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgbattn.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    inc = os.path.join(ROOT, "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def _source_list() -> str:
    return "\n".join(os.path.basename(f) for f in _sources())


def up_to_date(debug: bool = False) -> bool:
    lib, stamp = (LIB_DEBUG, os.path.join(BUILD_DEBUG, "sources.txt")) if debug else \
        (LIB, os.path.join(BUILD, "sources.txt"))
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        if f.read() != _source_list():       # a source was added or removed
            return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _sources() + _headers() + [__file__])


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(debug):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    flags = FLAGS + (["-DGBATTN_DEBUG_CHECKS"] if debug else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(os.path.join(bdir, "sources.txt"), "w") as f:
        f.write(_source_list())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv,
                debug="--debug" in sys.argv))
