"""Builds the CUDA library in-tree with nvcc for sm_103a (one translation unit)."""
from __future__ import annotations

import glob
import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmla_verify_attn.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]
_lock = threading.Lock()


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/mla_verify_attn.cu into _build/libmla_verify_attn.so."""
    with _lock:
        if not force and not is_stale():
            return LIB_PATH
        os.makedirs(OUT_DIR, exist_ok=True)
        tmp = LIB_PATH + ".%d.tmp" % os.getpid()
        cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", tmp,
               os.path.join(CSRC, "mla_verify_attn.cu")]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed (%d):\n%s\n%s" % (r.returncode, " ".join(cmd),
                                                              r.stderr[-4000:]))
        os.replace(tmp, LIB_PATH)
        if verbose:
            print(r.stderr)
        return LIB_PATH
