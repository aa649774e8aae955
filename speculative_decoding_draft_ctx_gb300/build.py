"""In-tree build of libdspark_ctx_kv.so for sm_103a (no cmake, no torch
extension machinery): the kernel TU is compiled by nvcc and the host TU by
g++ in parallel, then linked by nvcc against the static CUDA runtime."""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libdspark_ctx_kv.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
KERNEL_SRC = os.path.join(CSRC, "ctx_kv_kernel.cu")
TMA_SRC = os.path.join(CSRC, "ctx_kv_tma.cu")
QK_SRC = os.path.join(CSRC, "qk_insert_kernel.cu")
PROJ_SRC = os.path.join(CSRC, "proj_gemm.cu")
NORM_SRC = os.path.join(CSRC, "hidden_norm.cu")
GENERAL_SRC = os.path.join(CSRC, "ctx_kv_general.cu")
WARP_SRC = os.path.join(CSRC, "ctx_kv_warp.cu")
NOALLOC_SRC = os.path.join(CSRC, "ctx_kv_noalloc.cu")
CU_SRCS = (KERNEL_SRC, TMA_SRC, QK_SRC, PROJ_SRC, NORM_SRC, GENERAL_SRC, WARP_SRC, NOALLOC_SRC)
API_SRC = os.path.join(CSRC, "ctx_kv_api.cpp")
HEADERS = [os.path.join(CSRC, "ctx_kv_internal.h"), os.path.join(CSRC, "ctx_kv_device.cuh"),
           os.path.join(CSRC, "ctx_kv_pipe.cuh"),
           os.path.join(INCLUDE, "dspark_ctx_kv.h")]

_lock = threading.Lock()


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in [*CU_SRCS, API_SRC, *HEADERS])


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({' '.join(cmd)}):\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if a source is newer than it; returns its path."""
    with _lock:
        if not force and not _stale():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        home = cuda_home()
        nvcc = os.path.join(home, "bin", "nvcc")
        objs, cmds = [], []
        for src in CU_SRCS:
            obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
            cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            objs.append(obj)
            cmds.append(cmd)
        aobj = os.path.join(BUILD_DIR, "ctx_kv_api.o")
        cmds.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", os.path.join(home, "include"),
                     "-I", INCLUDE, "-c", API_SRC, "-o", aobj])
        objs.append(aobj)
        with ThreadPoolExecutor(len(cmds)) as ex:
            outs = list(ex.map(_run, cmds))
        if verbose:
            sys.stderr.write("".join(outs[:len(CU_SRCS)]))
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"])
        os.replace(tmp, LIB_PATH)
        return LIB_PATH


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB_PATH)
