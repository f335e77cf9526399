"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Each CUDA source compiles to an object in parallel (the decode kernels once
per cache format and head size), then nvcc links the
shared library (static CUDA runtime, no libcuda link: the tensor-map encoder
is looked up through the runtime's driver entry-point query).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkvq.so")
SOURCES = ["kvq_host.cu", "kvq_write.cu", "kvq_decode.cu", "kvq_decode_tc.cu", "kvq_decode_blk.cu",
           "kvq_static.cu", "kvq_calib.cu", "kvq_prefill.cu", "kvq_decode_variant.cu"]
HEADERS = ["kvq_common.cuh", "kvq_host.h", "kvq_decode.cuh", "kvq_tc.cuh", "kvq_decode_tc.cuh",
           "kvq_decode_blk.cuh", "kvq_prefill_tc.cuh"]
# (object, source, defines): one object per translation unit, the decode
# variants once per (format, head size); kvq_fmt 0 = BF16, 1 = E4M3, 2 = E5M2
UNITS = [(os.path.splitext(s)[0], s, []) for s in SOURCES if s != "kvq_decode_variant.cu"] + [
    (f"kvq_decode_f{fmt}_d{dh}", "kvq_decode_variant.cu",
     [f"-DKVQ_VARIANT_FMT={fmt}", f"-DKVQ_VARIANT_DH={dh}"])
    for fmt in (1, 2, 0) for dh in (128, 64)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    inc = os.path.join(os.path.dirname(HERE), "include", "kvq.h")
    return [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [inc, os.path.abspath(__file__)]


# The tests' timeout build: the same sources with the test hooks compiled in
# (a decode whose producer withholds one page on request) and bounded waits
# cut to 2^16 polls, in a directory of its own.  Never loaded by the package.
TEST_LIB = os.path.join(BUILD, "test", "libkvq_test.so")
TEST_DEFINES = ["-DKVQ_TEST_HOOKS", "-DKVQ_MAX_POLLS=65536u"]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build_test_lib(force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, extra=TEST_DEFINES, lib=TEST_LIB)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          lib: str = LIB) -> str:
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = list(extra or [])

    def compile_one(unit):
        name, src, defines = unit
        obj = os.path.join(out_dir, name + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *defines, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(UNITS), max(2, os.cpu_count() or 2))) as ex:
        objs = list(ex.map(compile_one, UNITS))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    ex = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else None
    print(build(force=True, verbose=v, extra=ex))
