"""Build and load the native library (libspec_verify.so, CUDA for sm_103a)."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
HEADER = os.path.join(ROOT, "include", "spec_verify.h")
LIB = os.path.join(PKG, "libspec_verify.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/spec_verify.cu into libspec_verify.so beside this file."""
    with _lock:
        stale = not os.path.exists(LIB) or any(
            os.path.getmtime(LIB) < os.path.getmtime(p) for p in (SRC, HEADER))
        if force or stale:
            tmp = LIB + f".tmp{os.getpid()}"
            cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            subprocess.check_call(cmd)
            os.replace(tmp, LIB)
    return LIB


def load() -> ctypes.CDLL:
    """Load the CUDA library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"native library {LIB} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB)
    vp, i, u, p = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.POINTER
    lib.spec_verify_init.restype = i
    lib.spec_verify_init.argtypes = [p(vp), i, i, i, i, u]
    lib.spec_verify.restype = i
    lib.spec_verify.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_lazy.restype = i
    lib.spec_verify_lazy.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_loss_grad.restype = i
    lib.spec_verify_loss_grad.argtypes = [vp, i, vp, vp, vp, i, vp, vp, vp, vp]
    lib.spec_verify_ex.restype = i
    lib.spec_verify_ex.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_noalloc.restype = i
    lib.spec_verify_noalloc.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_tv.restype = i
    lib.spec_verify_tv.argtypes = [vp, i, vp, vp, vp, vp, vp]
    lib.spec_verify_host.restype = i
    lib.spec_verify_host.argtypes = [vp, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.spec_verify_get_error.restype = i
    lib.spec_verify_get_error.argtypes = [vp, p(i)]
    lib.spec_verify_selftest_wait.restype = i
    lib.spec_verify_selftest_wait.argtypes = [vp, i, p(ctypes.c_longlong)]
    lib.spec_verify_info.restype = i
    lib.spec_verify_info.argtypes = [vp, p(i), p(i), p(i), p(i), p(i)]
    lib.spec_verify_kernel_times.restype = i
    lib.spec_verify_kernel_times.argtypes = [vp, vp, i, p(i)]
    lib.spec_verify_destroy.restype = None
    lib.spec_verify_destroy.argtypes = [vp]
    lib.spec_verify_strerror.restype = ctypes.c_char_p
    lib.spec_verify_strerror.argtypes = [i]
    _lib = lib
    return lib
