"""Build libfa_gb300.so in-tree with nvcc for sm_103a.

The three translation units compile in parallel, then link into one shared
library next to this file.  No CMake, no torch extension machinery.
"""
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libfa_gb300.so")
SOURCES = ["fa_api.cu", "fa_prefill.cu", "fa_decode.cu", "fa_decode_noalloc.cu",
           "fa_backward.cu", "fa_host.cu"]
HEADERS = ["fa_ptx.cuh", "fa_internal.h"]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", CSRC, "-I", INCLUDE]


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "fa.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    with tempfile.TemporaryDirectory(prefix="fa_build_") as tmp:
        procs, objs = [], []
        for s in SOURCES:
            obj = os.path.join(tmp, s.replace(".cu", ".o"))
            cmd = [NVCC] + ARCH + FLAGS + extra + ["-c", os.path.join(CSRC, s), "-o", obj]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                              stderr=subprocess.STDOUT, text=True)))
            objs.append(obj)
        failed = []
        for s, pr in procs:
            out, _ = pr.communicate()
            if out and (verbose or ptxas_info or pr.returncode):
                sys.stdout.write(out)
            if pr.returncode:
                failed.append(s)
        if failed:
            raise RuntimeError(f"nvcc failed for {failed}")
        tmp_lib = os.path.join(tmp, "libfa_gb300.so")
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp_lib] + objs
        subprocess.check_call(cmd)
        os.replace(tmp_lib, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv))
