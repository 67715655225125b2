"""Builds the CUDA library libpagedkv.so in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel; the result is linked with the
static CUDA runtime, so the library loads on machines without a GPU driver
(the driver is reached only when a call needs it).
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
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]
SOURCES = ["allocator.cpp", "prefix_cache.cpp", "pool.cu", "decode.cu", "vmm.cu", "prefill.cu",
           "cascade.cu", "tmap.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv.so")
    return path


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "paged_kv.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def _shared_inputs():
    """Headers every translation unit may include, and this script."""
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "paged_kv.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def _stale(src: str, shared_mtime: float) -> bool:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
    if not os.path.exists(obj):
        return True
    return os.path.getmtime(obj) < max(shared_mtime, os.path.getmtime(os.path.join(CSRC, src)))


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libpagedkv.so."""
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in _inputs())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    # recompile only the sources newer than their object (or all of them when
    # a shared header or this script changed)
    shared = max(os.path.getmtime(p) for p in _shared_inputs())
    todo = [s for s in SOURCES if force or verbose or _stale(s, shared)]
    with cf.ThreadPoolExecutor(max_workers=max(1, len(todo))) as ex:
        list(ex.map(lambda s: _compile(s, verbose), todo))
    objs = [os.path.join(OUT_DIR, s + ".o") for s in SOURCES]
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
