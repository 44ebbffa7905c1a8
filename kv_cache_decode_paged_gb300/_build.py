"""Build libkvattn.so in-tree with nvcc for sm_103a (GB300).

One nvcc process per translation unit, run in parallel, then a shared link.
The CUDA runtime is linked statically; the driver's tensor-map encoder is
reached through the runtime's entry-point query, so the library loads on a
machine without a GPU (for symbol checks) and links no libcuda.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvattn.so")
SOURCES = ["api.cu", "append.cu", "plan_combine.cu", "decode_gqa.cu", "decode_gqa_tc.cu",
           "decode_mla.cu", "noalloc.cu", "absorb.cu", "prefill_mla.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "kvattn.h"))
    files.append(os.path.abspath(__file__))
    return files


# Test-only variant: every main-loop mbarrier wait gives up after 2 ms (the
# exit-path drains keep their full limit), and CTA 0 of the GQA decode never
# signals chunk 3 of its walk, so that a wait runs out on the GPU and the abort
# path can be checked there.  Built on demand by its test, never by build().
WAIT_TEST_LIB = os.path.join(BUILD, "wait_test", "libkvattn_wait_test.so")
WAIT_TEST_DEFINES = ["-DKV_WAIT_NS=2000000ull", "-DKV_TEST_DROP_CHUNK=3"]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    # extra nvcc flags for tuning sweeps (e.g. -D overrides of kernel constants)
    extra = os.environ.get("KVATTN_NVCC_EXTRA", "").split()
    return _build_lib(LIB, BUILD, extra, force, verbose, ptxas_info)


def build_wait_test(force: bool = False) -> str:
    return _build_lib(WAIT_TEST_LIB, os.path.dirname(WAIT_TEST_LIB), WAIT_TEST_DEFINES, force)


def _build_lib(lib: str, build_dir: str, extra: list, force: bool = False, verbose: bool = False,
               ptxas_info: bool = False) -> str:
    if not force and not is_stale(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    exe = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + list(extra)

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [exe, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    tmp = lib + ".tmp"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
