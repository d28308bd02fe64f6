"""CPU oracle for speculative-decoding verification (fp64, plain C).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  It shares no code with
the CUDA library: the C source ``spec_verify_oracle.c`` restates the method
from the pages (sources and readings are in that file's header) and this
module only marshals numpy arrays into it.

Every function here is pinned by ``tests/test_oracle_*.py`` against properties
the pages fix (target preservation, acceptance = sum min(p, q) = 1 - TV,
p = q accepts everything, greedy = argmax match) and against closed forms and
library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
SOURCE = os.path.join(_HERE, "spec_verify_oracle.c")
_LIB_PATH = os.path.join(_BUILD, "libspec_verify_oracle.so")
_lock = threading.Lock()
_libs: dict[str, ctypes.CDLL] = {}

FP32 = 0
BF16 = 1
FP64 = 2   # single-row functions only (finite differences in the tests)
TIE_BAND = 1e-6


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library (gcc, -O2, fp64)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                           "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
            compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
    lib.so_argmax.restype = i64
    lib.so_argmax.argtypes = [vp, ctypes.c_int, i64]
    lib.so_log_softmax.restype = d
    lib.so_log_softmax.argtypes = [vp, ctypes.c_int, i64, d, vp]
    lib.so_accept.restype = ctypes.c_int
    lib.so_accept.argtypes = [d, d, d, ctypes.POINTER(ctypes.c_int)]
    lib.so_sample.restype = i64
    lib.so_sample.argtypes = [vp, i64, d, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)]
    lib.so_entropy.restype = d
    lib.so_entropy.argtypes = [vp, ctypes.c_int, i64, d]
    lib.so_entropy_batch.restype = ctypes.c_int
    lib.so_entropy_batch.argtypes = [i64, i32, i64, i32, vp, vp, vp, vp, vp, ctypes.c_int]
    lib.so_overlap_grad.restype = ctypes.c_int
    lib.so_overlap_grad.argtypes = [vp, vp, ctypes.c_int, i64, d, ctypes.c_int, d, vp, vp, vp, vp]
    lib.so_overlap_grad_batch.restype = ctypes.c_int
    lib.so_overlap_grad_batch.argtypes = [i64, i32, i64, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, ctypes.c_int]
    lib.so_verify_batch.restype = ctypes.c_int
    lib.so_verify_batch.argtypes = [i64, i32, i64, i32, vp, vp, vp, vp, vp, i32,
                                    vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """The oracle library (or another build of it, e.g. a planted-mistake copy)."""
    key = path or _LIB_PATH
    with _lock:
        lib = _libs.get(key)
    if lib is None:
        if path is None:
            build()
        lib = _bind(ctypes.CDLL(key))
        with _lock:
            _libs[key] = lib
    return lib


class Oracle:
    """numpy-facing wrapper over one build of the oracle library."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    @staticmethod
    def _row(z, dtype):
        a = np.ascontiguousarray(z, dtype={FP32: np.float32, BF16: np.uint16, FP64: np.float64}[dtype])
        return a

    def argmax(self, z, dtype: int = FP32) -> int:
        a = self._row(z, dtype)
        return int(self.lib.so_argmax(a.ctypes.data, dtype, a.shape[-1]))

    def log_softmax(self, z, T: float, dtype: int = FP32):
        """(log p, lse) of one row at temperature T > 0."""
        a = self._row(z, dtype)
        out = np.empty(a.shape[-1], np.float64)
        lse = self.lib.so_log_softmax(a.ctypes.data, dtype, a.shape[-1], float(T), out.ctypes.data)
        return out, float(lse)

    def probs(self, z, T: float, dtype: int = FP32) -> np.ndarray:
        """The row's distribution at temperature T (one-hot argmax at T == 0)."""
        if T == 0:
            p = np.zeros(np.shape(z)[-1])
            p[self.argmax(z, dtype)] = 1.0
            return p
        lp, _ = self.log_softmax(z, T, dtype)
        return np.exp(lp)

    def entropy(self, z, T: float, dtype: int = FP32) -> float:
        """Entropy (nats) of one row's distribution at temperature T (0 at T == 0)."""
        a = self._row(z, dtype)
        return float(self.lib.so_entropy(a.ctypes.data, dtype, a.shape[-1], float(T)))

    def entropy_batch(self, target, draft, temperature, dtype: int, nthreads: int = 1):
        """Entropies of every target row [B,k+1] and draft row [B,k] (fp64)."""
        tgt = self._row(target, dtype)
        dft = self._row(draft, dtype)
        B, k1, V = tgt.shape
        k = k1 - 1
        assert dft.shape == (B, k, V)
        T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
        ent_t = np.empty((B, k + 1))
        ent_d = np.empty((B, k))
        rc = self.lib.so_entropy_batch(B, k, V, dtype, tgt.ctypes.data, dft.ctypes.data, T.ctypes.data,
                                       ent_t.ctypes.data, ent_d.ctypes.data, int(nthreads))
        if rc != 0:
            raise ValueError(f"so_entropy_batch failed: {rc}")
        return ent_t, ent_d

    def overlap_grad(self, zt, zd, T: float, kind: int, w: float = 1.0, dtype: int = FP32):
        """(loss, alpha, grad [V], tie mass) of one position: kind 0 = TV loss 1 - alpha,
        kind 1 = overlap loss -ln alpha; grad is d(w * loss)/d(draft logits)."""
        a, b = self._row(zt, dtype), self._row(zd, dtype)
        V = a.shape[-1]
        loss, alpha, tie = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        g = np.empty(V)
        self.lib.so_overlap_grad(a.ctypes.data, b.ctypes.data, dtype, V, float(T), int(kind), float(w),
                                 ctypes.byref(loss), ctypes.byref(alpha), g.ctypes.data, ctypes.byref(tie))
        return loss.value, alpha.value, g, tie.value

    def overlap_grad_batch(self, target, draft, temperature, kind: int, weights=None, dtype: int = FP32,
                           nthreads: int = 1) -> dict:
        """Losses and draft-logit gradients of every position of a batch (fp64)."""
        tgt, dft = self._row(target, dtype), self._row(draft, dtype)
        B, k1, V = tgt.shape
        k = k1 - 1
        T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
        w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32).reshape(B, k)
        out = dict(loss=np.empty((B, k)), alpha=np.empty((B, k)), grad=np.empty((B, k, V)), tie=np.empty((B, k)))
        rc = self.lib.so_overlap_grad_batch(B, k, V, dtype, tgt.ctypes.data, dft.ctypes.data, T.ctypes.data, int(kind),
                                            None if w is None else w.ctypes.data, out["loss"].ctypes.data,
                                            out["alpha"].ctypes.data, out["grad"].ctypes.data, out["tie"].ctypes.data,
                                            int(nthreads))
        if rc != 0:
            raise ValueError(f"so_overlap_grad_batch failed: {rc}")
        return out

    def accept(self, lp: float, lq: float, u: float):
        tie = ctypes.c_int(0)
        acc = self.lib.so_accept(float(lp), float(lq), float(u), ctypes.byref(tie))
        return bool(acc), bool(tie.value)

    def sample(self, w, u: float):
        a = np.ascontiguousarray(w, dtype=np.float64)
        tie = ctypes.c_int(0)
        tot = ctypes.c_double(0)
        y = self.lib.so_sample(a.ctypes.data, a.shape[-1], float(u), ctypes.byref(tie), ctypes.byref(tot))
        return int(y), bool(tie.value), float(tot.value)

    def verify(self, target, draft, tokens, temperature, uniforms, dtype: int, want_tv: bool = True,
               nthreads: int = 1) -> dict:
        """Verify B chains.  target [B,k+1,V], draft [B,k,V] (fp32 or bf16 bits),
        tokens [B,k] int32, temperature [B], uniforms [B,k+1]."""
        tgt = self._row(target, dtype)
        dft = self._row(draft, dtype)
        B, k1, V = tgt.shape
        k = k1 - 1
        assert dft.shape == (B, k, V)
        x = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, k)
        T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
        u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, k + 1)
        out = dict(
            tokens=np.empty((B, k + 1), np.int32), tau=np.empty(B, np.int32),
            p_draft=np.empty((B, k)), q_draft=np.empty((B, k)), tv=np.full((B, k), np.nan),
            accept_tie=np.zeros((B, k), np.int32), cdf_tie=np.zeros(B, np.int32),
            residual_fallback=np.zeros(B, np.int32), residual_mass=np.zeros(B),
        )
        rc = self.lib.so_verify_batch(B, k, V, dtype, tgt.ctypes.data, dft.ctypes.data, x.ctypes.data,
                                      T.ctypes.data, u.ctypes.data, int(bool(want_tv)),
                                      out["tokens"].ctypes.data, out["tau"].ctypes.data,
                                      out["p_draft"].ctypes.data, out["q_draft"].ctypes.data,
                                      out["tv"].ctypes.data, out["accept_tie"].ctypes.data,
                                      out["cdf_tie"].ctypes.data, out["residual_fallback"].ctypes.data,
                                      out["residual_mass"].ctypes.data, int(nthreads))
        if rc != 0:
            raise ValueError(f"so_verify_batch failed: {rc}")
        return out


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
