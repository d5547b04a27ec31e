"""Build libdsa.so in-tree with nvcc for sm_103a (one -gencode, translation units in parallel).

build(checked=True) builds libdsa_checked.so instead: the same sources with -DDSA_CHECKED, whose kernels also
bounds-check their computed shared-memory and table indexes (a bad index records DSA_ERR_DEVICE_FAULT and the
access is skipped).  The binding loads it when the environment sets DSA_CHECKED=1."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdsa.so")
LIB_CHECKED = os.path.join(PKG, "libdsa_checked.so")
SOURCES = ["api.cu", "compress.cu", "index_scores.cu", "topk.cu", "attention.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa.so")


def _cuda_lib_dir(nvcc):
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _flags():
    return ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *ARCH]


def build(verbose=False, ptxas_verbose=False, checked=False):
    """Compile every CUDA source and link libdsa.so (or libdsa_checked.so); returns its path.  Rebuilds only
    when stale."""
    nvcc = _nvcc()
    lib = LIB_CHECKED if checked else LIB
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dsa.h"), __file__]
    newest = max(os.path.getmtime(d) for d in deps)
    if os.path.exists(lib) and os.path.getmtime(lib) >= newest and not ptxas_verbose:
        return lib

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *_flags(), *(["-DDSA_CHECKED"] if checked else []), "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stdout + res.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv, checked="--checked" in sys.argv))
