"""Builds libbst.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery): one object per translation unit, compiled in parallel,
then linked into a shared library with the CUDA runtime linked statically."""
import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libbst.so")
UNITS = ["api.cu", "gemm_dense.cu", "gemm_pair.cu", "gemm_mxf8.cu", "gemm_quant.cu", "sched_map.cu", "noalloc.cu", "slice_k.cu"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "bst.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _sources())


def _flags():
    return [GENCODE, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def build(force=False, verbose=False, ptxas_info=False):
    """Compile every unit and link libbst.so.  Returns the library path."""
    if not force and not stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    flags = _flags() + (["-Xptxas", "-v"] if ptxas_info else [])

    def compile_one(unit):
        obj = os.path.join(OUT_DIR, unit.replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", os.path.join(CSRC, unit), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (unit, " ".join(cmd), r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_one, UNITS))
    if verbose or ptxas_info:
        for obj, err in results:
            if err.strip():
                print("== %s\n%s" % (os.path.basename(obj), err))
    tmp = LIB + ".tmp"
    cmd = [cc, GENCODE, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
