"""Build libfp8bs.so in-tree from csrc/*.cu with nvcc for sm_103a only.

Each translation unit compiles in parallel; the objects link into one shared
library with the CUDA runtime linked statically, so the library needs only the
driver at load time. Run as a script or call build().
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp8bs.so")
# the same library with every plain global store of its kernels bounds-checked
# (-DFP8BS_CHECK; see csrc/check.cuh): a test build, not the product path
CHECK_LIB = os.path.join(HERE, "libfp8bs_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division/sqrt and no flush-to-zero: the scales must round exactly like
# the reference definition (no fast-math anywhere).
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-ftz=false", "-prec-div=true",
           "-prec-sqrt=true", "-fmad=true", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fp8bs.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, check: bool = False) -> str:
    """Build libfp8bs.so (or, with check=True, libfp8bs_check.so); returns its path."""
    lib = CHECK_LIB if check else LIB
    if not force and up_to_date(lib):
        return lib
    bdir = os.path.join(BUILD_DIR, "check") if check else BUILD_DIR
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DFP8BS_CHECK"] if check else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVFLAGS, *extra, "-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, p.stdout, p.stderr))
        if verbose_ptxas:
            sys.stderr.write(p.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(sources())) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (p.stdout, p.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="-v" in sys.argv, check="--check" in sys.argv))
