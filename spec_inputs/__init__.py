"""Seeded synthetic inputs for speculative-decoding verification.

Shared by the CPU oracle's tests, the CUDA library's tests and the benchmark.
It holds input generation only (Philox4x32-10 uniforms, Box-Muller normals,
bf16 rounding, Gumbel-max draft sampling); none of the verification
arithmetic lives here.  The C source is ``gen.c`` beside this file; it is
compiled on first use (or by ``build()``) into ``_build/libspec_inputs.so``.

Workload presets follow the five verification workloads this library is
measured on (chains B, draft length k, vocabulary V, logit dtype, logit
distributions and temperatures); ``Workload.scaled`` keeps a recipe and
shrinks B or V for fast tests.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libspec_inputs.so")
_lock = threading.Lock()
_lib = None

FP32 = 0
BF16 = 1

STREAM_TARGET, STREAM_DRAFT, STREAM_GUMBEL, STREAM_VERIFY, STREAM_BOOST, STREAM_TEMP = range(6)


class _Workload(ctypes.Structure):
    _fields_ = [
        ("seed", ctypes.c_uint64),
        ("k", ctypes.c_int32),
        ("vocab", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("batch_total", ctypes.c_int32),
        ("sigma_a", ctypes.c_double),
        ("sigma_b", ctypes.c_double),
        ("split", ctypes.c_int32),
        ("n_boost", ctypes.c_int32),
        ("boost", ctypes.c_double),
        ("draft_mode", ctypes.c_int32),
        ("draft_sigma", ctypes.c_double),
        ("temp_mode", ctypes.c_int32),
        ("temp_lo", ctypes.c_double),
        ("temp_hi", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libspec_inputs.so (plain C, no GPU)."""
    src = os.path.join(_HERE, "gen.c")
    with _lock:
        if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                                   "-o", tmp, src, "-lm"])
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.sg_generate.restype = ctypes.c_int
        lib.sg_generate.argtypes = [ctypes.POINTER(_Workload), ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.sg_uniform.restype = ctypes.c_float
        lib.sg_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64]
        lib.sg_uniforms.restype = None
        lib.sg_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        lib.sg_philox4x32_10.restype = None
        lib.sg_philox4x32_10.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.sg_f32_to_bf16.restype = ctypes.c_uint16
        lib.sg_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.sg_gumbel_argmax_rows.restype = None
        lib.sg_gumbel_argmax_rows.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_uint64, ctypes.c_void_p]
        _lib = lib
    return _lib


@dataclasses.dataclass(frozen=True)
class Workload:
    """One verification workload: B chains of k drafts over a V-token vocabulary."""
    name: str
    batch: int
    k: int
    vocab: int
    dtype: int                  # FP32 or BF16
    sigma_a: float              # target logit scale (chains b < split)
    sigma_b: float = 0.0        # target logit scale (chains b >= split)
    split: int | None = None    # None: every chain uses sigma_a
    n_boost: int = 0            # distinct boosted ids per target row
    boost: float = 0.0          # value added to boosted ids
    draft_mode: int = 0         # 0: target + N(0, draft_sigma^2); 1: independent N(0, draft_sigma^2)
    draft_sigma: float = 1.0
    temp_mode: int = 0          # 0: fixed temp_lo; 1: per chain U[temp_lo, temp_hi]
    temp_lo: float = 1.0
    temp_hi: float = 1.0
    want_tv: bool = False
    seed: int = 0

    @property
    def itemsize(self) -> int:
        return 4 if self.dtype == FP32 else 2

    @property
    def logit_bytes(self) -> int:
        """Bytes of target + draft logits: B * (2k+1) * V * s."""
        return self.batch * (2 * self.k + 1) * self.vocab * self.itemsize

    def scaled(self, batch: int | None = None, vocab: int | None = None, name: str | None = None,
               seed: int | None = None) -> "Workload":
        b = self.batch if batch is None else batch
        split = self.split
        if split is not None:
            split = max(0, min(b, (split * b) // self.batch))
        return dataclasses.replace(self, batch=b, vocab=self.vocab if vocab is None else vocab,
                                   split=split, name=name or f"{self.name}@B{b}V{vocab or self.vocab}",
                                   seed=self.seed if seed is None else seed)

    def _c(self) -> _Workload:
        split = self.batch if self.split is None else self.split
        return _Workload(self.seed, self.k, self.vocab, self.dtype, self.batch, self.sigma_a,
                         self.sigma_b, split, self.n_boost, self.boost, self.draft_mode,
                         self.draft_sigma, self.temp_mode, self.temp_lo, self.temp_hi)


# The five verification workloads (synthetic stand-ins for the pages' coding and
# validation workloads, which are not available).
TINY = Workload("tiny_b1_k3_v16_fp32", 1, 3, 16, FP32, 2.0, draft_sigma=0.5)
C2 = Workload("b8_k7_v32000_fp32", 8, 7, 32000, FP32, 2.0, draft_sigma=0.7)
C3_T0 = Workload("b64_k7_v151552_bf16_t0", 64, 7, 151552, BF16, 3.0, n_boost=20, boost=8.0,
                 draft_sigma=1.0, temp_lo=0.0, temp_hi=0.0)
C3_T06 = dataclasses.replace(C3_T0, name="b64_k7_v151552_bf16_t0.6", temp_lo=0.6, temp_hi=0.6)
C3_T1 = dataclasses.replace(C3_T0, name="b64_k7_v151552_bf16_t1", temp_lo=1.0, temp_hi=1.0)
C4 = Workload("b256_k15_v151552_bf16_mixed", 256, 15, 151552, BF16, 6.0, sigma_b=0.5, split=128,
              draft_sigma=1.0, temp_mode=1, temp_lo=0.3, temp_hi=1.2)
C5 = Workload("b1024_k7_v151552_bf16_indep_tv", 1024, 7, 151552, BF16, 2.0, draft_mode=1,
              draft_sigma=2.0, want_tv=True)

WORKLOADS = {w.name: w for w in (TINY, C2, C3_T0, C3_T06, C3_T1, C4, C5)}


@dataclasses.dataclass
class Batch:
    """Host-side inputs of chains [b0, b0 + nb) of a workload."""
    workload: Workload
    b0: int
    target: np.ndarray       # [nb, k+1, V] float32 or uint16 (bf16 bits)
    draft: np.ndarray        # [nb, k, V]
    tokens: np.ndarray       # [nb, k] int32
    temperature: np.ndarray  # [nb] float32
    uniforms: np.ndarray     # [nb, k+1] float32

    @property
    def nb(self) -> int:
        return self.target.shape[0]


def empty_logits(shape, dtype: int) -> np.ndarray:
    return np.empty(shape, dtype=np.float32 if dtype == FP32 else np.uint16)


def generate(w: Workload, b0: int = 0, nb: int | None = None, nthreads: int | None = None,
             out: dict | None = None) -> Batch:
    """Generate chains [b0, b0+nb) of workload w (all chains by default).

    ``out`` may supply preallocated arrays (e.g. pinned host memory viewed as
    numpy) under the keys target/draft/tokens/temperature/uniforms.
    """
    lib = _load()
    if nb is None:
        nb = w.batch - b0
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    out = out or {}
    tgt = out.get("target")
    if tgt is None:
        tgt = empty_logits((nb, w.k + 1, w.vocab), w.dtype)
    dft = out.get("draft")
    if dft is None:
        dft = empty_logits((nb, w.k, w.vocab), w.dtype)
    tok = out.get("tokens")
    if tok is None:
        tok = np.empty((nb, w.k), np.int32)
    tmp = out.get("temperature")
    if tmp is None:
        tmp = np.empty((nb,), np.float32)
    uni = out.get("uniforms")
    if uni is None:
        uni = np.empty((nb, w.k + 1), np.float32)
    for a in (tgt, dft, tok, tmp, uni):
        assert a.flags["C_CONTIGUOUS"]
    cw = w._c()
    rc = lib.sg_generate(ctypes.byref(cw), b0, nb, tgt.ctypes.data, dft.ctypes.data, tok.ctypes.data,
                         tmp.ctypes.data, uni.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError(f"sg_generate failed with code {rc}")
    return Batch(w, b0, tgt, dft, tok, tmp, uni)


def uniform(seed: int, stream: int, row: int, col: int) -> float:
    return float(_load().sg_uniform(seed, stream, row, col))


def uniforms(seed: int, stream: int, row0: int, n_rows: int, n_cols: int) -> np.ndarray:
    out = np.empty((n_rows, n_cols), np.float32)
    _load().sg_uniforms(seed, stream, row0, n_rows, n_cols, out.ctypes.data)
    return out


def philox4x32_10(counter, key) -> np.ndarray:
    c = np.asarray(counter, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.empty(4, np.uint32)
    _load().sg_philox4x32_10(c.ctypes.data, k.ctypes.data, o.ctypes.data)
    return o


def f32_to_bf16(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even); returns the bf16 bit patterns."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    flat = np.array([lib.sg_f32_to_bf16(float(v)) for v in a.ravel()], dtype=np.uint16)
    return flat.reshape(a.shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def gumbel_argmax(seed: int, logits: np.ndarray, dtype: int, temps: np.ndarray, row0: int = 0) -> np.ndarray:
    """Draw one token per row from softmax(logits / T) with the Gumbel-max trick."""
    lib = _load()
    z = np.ascontiguousarray(logits)
    rows = int(np.prod(z.shape[:-1]))
    V = z.shape[-1]
    t = np.ascontiguousarray(np.broadcast_to(np.asarray(temps, np.float32), (rows,)))
    out = np.empty(rows, np.int32)
    lib.sg_gumbel_argmax_rows(seed, z.ctypes.data, dtype, rows, V, t.ctypes.data, row0, out.ctypes.data)
    return out.reshape(z.shape[:-1])
