"""In-tree build of libdsa_mla.so (sm_103a) with nvcc.

Each translation unit under csrc/ is compiled in parallel to an object in _build/, then
linked into sparse_mla_paged_gb300/libdsa_mla.so against the shared CUDA runtime (and
cuBLAS, for the load-time absorb GEMMs).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdsa_mla.so")
SOURCES = ["api.cu", "prologue.cu", "decode.cu", "combine.cu", "static_scratch.cu", "latent_write.cu", "select.cu",
           "absorb.cu"]
# Translation units: (source, object, extra flags); decode.cu is built once per tile size.
UNITS = [("api.cu", "api.o", []), ("prologue.cu", "prologue.o", []),
         ("decode.cu", "decode64.o", ["-DDSA_TILE=64"]), ("decode.cu", "decode128.o", ["-DDSA_TILE=128"]),
         ("combine.cu", "combine.o", []), ("static_scratch.cu", "static_scratch.o", []),
         ("latent_write.cu", "latent_write.o", []), ("select.cu", "select.o", []), ("absorb.cu", "absorb.o", [])]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found")
    return p


def _compile(unit, extra: list[str]) -> str:
    src, obj_name, flags = unit
    obj = os.path.join(BUILD, obj_name)
    cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           "-I", CSRC, *flags, "-c", os.path.join(CSRC, src), "-o", obj, *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dsa_mla.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (if sources changed) and return the path of libdsa_mla.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(lambda u: _compile(u, extra), UNITS))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-lcublas"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
