"""Builds libqp.so in-tree with nvcc for sm_103a (no torch extension machinery:
the library is a plain C-ABI shared object)."""
import concurrent.futures
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC,
                 "-ftz=false", "-prec-div=true", "-prec-sqrt=true"]
# Per-file extra flags: the standalone dequant is compiled without FMA
# contraction (its products are exact anyway; this keeps every operation
# rounded on its own, as the oracle is).
SOURCES = {
    "api.cu": [],
    "dequant.cu": ["-fmad=false"],
    "qgemm.cu": [],
    "gemv.cu": [],
}


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "qp.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force=False, verbose_ptxas=False):
    """Compile every translation unit in parallel and link libqp.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(name):
        obj = os.path.join(BUILD, name + ".o")
        cmd = [nvcc] + COMMON + SOURCES[name] + extra + ["-c", os.path.join(CSRC, name), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (name, r.stdout, r.stderr))
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    if verbose_ptxas:
        for _, log in results:
            print(log)
    return LIB
