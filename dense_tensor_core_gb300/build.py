"""Build the CUDA library in-tree: dense_tensor_core_gb300/libdtc_gemm.so (sm_103a only).

One translation unit per kernel family plus the API unit, compiled in parallel with nvcc (one
-gencode), then linked into one shared library. The CUDA runtime is linked statically so the
library loads without a GPU (the CPU tests check its exports) and carries no rpath.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libdtc_gemm.so")
OBJ_DIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cand, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def _inputs():
    files = sources() + [os.path.join(INCLUDE, "dtc_gemm.h")]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return files


def _compile(src, obj_dir, verbose_ptxas):
    obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           "-I", CSRC, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.check_call(cmd)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(f) for f in _inputs())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = sources()
    # objects in a directory of this build's own, so concurrent builds cannot mix their files
    with tempfile.TemporaryDirectory(dir=OBJ_DIR) as obj_dir:
        with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
            objs = list(ex.map(lambda s: _compile(s, obj_dir, verbose_ptxas), srcs))
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
