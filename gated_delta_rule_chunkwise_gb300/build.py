"""Build libldn.so (the CUDA library behind include/ldn.h) for sm_103a.

Each .cu file directly under csrc/ is compiled by its own nvcc process (in
parallel), then the objects are linked into lib/libldn.so inside the package.
The diagnostic kernels (csrc/diag/, include/ldn_diag.h) are linked into a
library of their own, lib/libldn_diag.so, which only the tests load.  The CUDA
runtime is linked statically, so the libraries need only the driver at run
time.  Nothing here runs at import time; __graft_entry__.build() and the
tests call build().
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libldn.so")
DIAG_DIR = os.path.join(CSRC, "diag")
DIAG_LIB_PATH = os.path.join(LIB_DIR, "libldn_diag.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libldn")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _diag_sources():
    return sorted(os.path.join(DIAG_DIR, f) for f in os.listdir(DIAG_DIR) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _stamp() -> str:
    h = hashlib.sha256()
    for p in _sources() + _diag_sources() + _headers():
        with open(p, "rb") as f:
            h.update(p.encode() + f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def _compile(nvcc, src, log_dir):
    tag = "diag_" if os.path.dirname(src) == DIAG_DIR else ""
    obj = os.path.join(OBJ_DIR, tag + os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(log_dir, os.path.basename(src) + ".log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-6000:]}")
    return obj


def _link(nvcc, objs, path):
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(path)} failed:\n{r.stderr[-6000:]}")
    os.replace(tmp, path)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libldn.so and libldn_diag.so if any source changed;
    return the path of libldn.so."""
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    stamp_file = os.path.join(OBJ_DIR, "stamp")
    stamp = _stamp()
    if (not force and os.path.exists(LIB_PATH) and os.path.exists(DIAG_LIB_PATH) and
            os.path.exists(stamp_file)):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB_PATH
    nvcc = _nvcc()
    srcs, dsrcs = _sources(), _diag_sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs) + len(dsrcs))) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, OBJ_DIR), srcs + dsrcs))
    _link(nvcc, objs[:len(srcs)], LIB_PATH)
    _link(nvcc, objs[len(srcs):], DIAG_LIB_PATH)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    if verbose:
        for s in srcs + dsrcs:
            with open(os.path.join(OBJ_DIR, os.path.basename(s) + ".log")) as f:
                print(f.read())
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
