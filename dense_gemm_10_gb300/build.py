"""Build the sm_103a GEMM library in-tree: dense_gemm_10_gb300/libgemm_gb300.so.

Each CUDA translation unit is compiled by nvcc in parallel (one -gencode for
sm_103a), then linked into one shared library with the CUDA runtime linked
statically, so the library loads on a machine without a GPU (its entry points
then report GEMM_ERR_NO_DEVICE).  ptxas register / spill reports are kept next
to the objects in _build/*.ptxas.log.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libgemm_gb300.so")
HEADER = os.path.join(ROOT, "include", "gemm_gb300.h")

SOURCES = ["gemm_api.cu", "tc_dispatch.cu", "aux_kernels.cu", "probe.cu",
           # one translation unit per kernel configuration: tile width, CTA group, input kind
           "tc_gemm_bn64_cg1.cu", "tc_gemm_bn128_cg1.cu", "tc_gemm_bn256_cg1.cu", "tc_gemm_bn64_cg2.cu",
           "tc_gemm_bn128_cg2.cu", "tc_gemm_bn256_cg2.cu",
           "tc_gemm_bn64_cg1_f8.cu", "tc_gemm_bn128_cg1_f8.cu", "tc_gemm_bn128_cg2_f8.cu", "tc_gemm_bn256_cg2_f8.cu",
           "tc_gemm_bn64_cg1_tf32.cu", "tc_gemm_bn128_cg1_tf32.cu", "tc_gemm_bn256_cg2_tf32.cu",
           "tc_gemm_bn64_cg1_dq.cu", "tc_gemm_bn256_cg2_ew8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build the GEMM library")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [HEADER, os.path.abspath(__file__)]


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _compile(nvcc, src):
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if not _stale(obj, [path] + _deps()):
        return obj
    cmd = [nvcc] + ARCH + FLAGS + ["-c", path, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".ptxas.log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr[-4000:]))
    os.replace(obj + ".tmp", obj)
    return obj


def build(force=False, verbose=False):
    """Compile (if stale) and link the library; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force:
        for f in os.listdir(BUILD_DIR):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD_DIR, f))
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s), SOURCES))
    if force or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s" % r.stderr[-4000:])
        os.replace(tmp, LIB_PATH)
    if verbose:
        print(LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
