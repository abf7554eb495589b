"""Builds the CUDA library ``_lib/libmla_dcp.so`` for sm_103a (in-tree).

Each translation unit is compiled in parallel with one ``-gencode`` and the
objects are linked into one shared library with the CUDA runtime linked
statically, so the library loads on a machine without a GPU driver (the
driver is looked up at first use).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libmla_dcp.so")
SOURCES = ["partial.cu", "partial_fp8.cu", "wuv_gemm.cu", "plan_merge.cu", "combine.cu", "capi.cu", "noalloc.cu", "gqa.cu"]
HEADERS = ["common.cuh", "merge.cuh", "ptx.cuh", "host_util.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = os.path.join(cuda, "bin", "nvcc")
    return exe if os.path.exists(exe) else (shutil.which("nvcc") or "nvcc")


INCLUDE = os.path.join(os.path.dirname(HERE), "include")


def flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I" + INCLUDE, *extra]


def _inputs():
    root = os.path.dirname(HERE)
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(root, "include", "mla_dcp.h")])


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force=False, verbose=False, extra_flags=()):
    if not (force or needs_build()):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = [os.path.join(OUT_DIR, os.path.splitext(s)[0] + ".o") for s in SOURCES]

    def compile_one(src, obj):
        cmd = [nvcc(), *flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(compile_one, SOURCES, objs))
    if verbose:
        for log in logs:
            if log.strip():
                print(log)
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", LIB, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return LIB


if __name__ == "__main__":
    import sys
    extra = ["-Xptxas", "-v"] if "-v" in sys.argv else []
    print(build(force=True, verbose=bool(extra), extra_flags=extra))
