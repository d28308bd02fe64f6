"""GB300-native speculative-decoding verification by rejection sampling.

A thin Python binding over the C-ABI library ``libspec_verify.so`` (see
``include/spec_verify.h``).  It only marshals arguments: every step of the
verification runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.

    sv = SpecVerifier(max_batch=1024, k=7, vocab=151552, dtype=torch.bfloat16)
    out = sv.verify(target, draft, tokens, temperature, uniforms, want_tv=True)
    out["tokens"], out["tau"], out["tv"]
"""
from __future__ import annotations

import ctypes

from . import _native

SV_OK, SV_ERR_ARG, SV_ERR_DTYPE, SV_ERR_SIZE, SV_ERR_CUDA, SV_ERR_ALLOC, SV_ERR_DATA, SV_ERR_TIMEOUT = range(8)
SV_FP32, SV_BF16 = 0, 1
SV_FLAG_HOST_STAGING, SV_FLAG_NO_TMA, SV_FLAG_KERNEL_TIMING = 1, 2, 4
SV_LOSS_TV, SV_LOSS_OVERLAP = 0, 1

build = _native.build


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _native.load().spec_verify_strerror(code).decode()
        super().__init__(f"{where}: {msg} (status {code})")
        self.code = code


def _check(code: int, where: str):
    if code != SV_OK:
        raise SpecVerifyError(code, where)


def _dtype_code(dtype) -> int:
    import torch
    if dtype in (torch.bfloat16, "bf16", "bfloat16", SV_BF16):
        return SV_BF16
    if dtype in (torch.float32, "fp32", "float32", SV_FP32):
        return SV_FP32
    raise ValueError(f"unsupported logit dtype {dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------- argument checks
# The library sees raw pointers and cannot tell a buffer's size, so every
# tensor is checked here, before the call: a wrong shape would otherwise make
# the kernels read or write past the end of a buffer.  These raise ValueError
# (not assert, which python -O removes).

def _check_tensor(t, name: str, dtype, shape: tuple, device):
    """t must have this dtype and shape, be contiguous, and live on `device`
    (a torch.device; for CUDA, the same index)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.type != device.type or (device.type == "cuda" and t.device.index != device.index):
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def check_batch(k: int, vocab: int, logit_dtype, max_batch: int, device, target, draft, tokens=None,
                temperature=None, uniforms=None, need_tokens: bool = True, need_uniforms: bool = True) -> int:
    """Checks a batch of inputs against a handle's k, vocabulary, dtype and
    capacity; returns the batch size B."""
    import torch
    if target is None or target.dim() != 3:
        raise ValueError("target must be a [B, k+1, V] tensor")
    B = int(target.shape[0])
    if B > max_batch:
        raise ValueError(f"batch {B} exceeds the handle's max_batch {max_batch}")
    _check_tensor(target, "target", logit_dtype, (B, k + 1, vocab), device)
    _check_tensor(draft, "draft", logit_dtype, (B, k, vocab), device)
    if need_tokens:
        _check_tensor(tokens, "tokens", torch.int32, (B, k), device)
    _check_tensor(temperature, "temperature", torch.float32, (B,), device)
    if need_uniforms:
        _check_tensor(uniforms, "uniforms", torch.float32, (B, k + 1), device)
    return B


def output_shapes(B: int, k: int, vocab: int, logit_dtype) -> dict:
    """dtype and shape of every output tensor an entry point may write."""
    import torch
    f32, i32 = torch.float32, torch.int32
    return {"tokens": (i32, (B, k + 1)), "tau": (i32, (B,)), "p_draft": (f32, (B, k)), "q_draft": (f32, (B, k)),
            "tv": (f32, (B, k)), "entropy_target": (f32, (B, k + 1)), "entropy_draft": (f32, (B, k)),
            "loss": (f32, (B, k)), "grad": (logit_dtype, (B, k, vocab))}


def check_outputs(out: dict, B: int, k: int, vocab: int, logit_dtype, device, required=("tokens", "tau")):
    """Checks the output tensors present in `out` (and that `required` are)."""
    shapes = output_shapes(B, k, vocab, logit_dtype)
    for name in required:
        if out.get(name) is None:
            raise ValueError(f"output {name} is required")
    for name, t in out.items():
        if t is None:
            continue
        if name not in shapes:
            raise ValueError(f"unknown output {name}")
        dtype, shape = shapes[name]
        _check_tensor(t, f"output {name}", dtype, shape, device)


class SpecVerifier:
    """One library handle: chains of k drafts over a vocabulary of `vocab` tokens."""

    def __init__(self, max_batch: int, k: int, vocab: int, dtype, flags: int = 0):
        self._lib = _native.load()
        self.max_batch, self.k, self.vocab = max_batch, k, vocab
        self.dtype_code = _dtype_code(dtype)
        self.flags = flags
        h = ctypes.c_void_p()
        _check(self._lib.spec_verify_init(ctypes.byref(h), max_batch, k, vocab, self.dtype_code, flags),
               "spec_verify_init")
        self._h = h
        import torch
        self.device = torch.device("cuda", torch.cuda.current_device())   # the handle's GPU

    @property
    def torch_dtype(self):
        import torch
        return torch.bfloat16 if self.dtype_code == SV_BF16 else torch.float32

    def close(self):
        if getattr(self, "_h", None):
            self._lib.spec_verify_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> dict:
        vals = [ctypes.c_int() for _ in range(5)]
        _check(self._lib.spec_verify_info(self._h, *[ctypes.byref(v) for v in vals]), "spec_verify_info")
        keys = ("cluster_size", "n_clusters", "rounds", "tma", "launches_per_call")
        return {k: v.value for k, v in zip(keys, vals)}

    @staticmethod
    def _stream(stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return ctypes.c_void_p(stream.cuda_stream)

    def alloc_outputs(self, batch: int, want_pq: bool = True, want_tv: bool = False, device="cuda",
                      want_entropy: bool = False) -> dict:
        import torch
        k = self.k
        out = {"tokens": torch.empty((batch, k + 1), dtype=torch.int32, device=device),
               "tau": torch.empty((batch,), dtype=torch.int32, device=device)}
        if want_pq:
            out["p_draft"] = torch.empty((batch, k), dtype=torch.float32, device=device)
            out["q_draft"] = torch.empty((batch, k), dtype=torch.float32, device=device)
        if want_tv:
            out["tv"] = torch.empty((batch, k), dtype=torch.float32, device=device)
        if want_entropy:
            out["entropy_target"] = torch.empty((batch, k + 1), dtype=torch.float32, device=device)
            out["entropy_draft"] = torch.empty((batch, k), dtype=torch.float32, device=device)
        return out

    def _check_inputs(self, target, draft, tokens, temperature, uniforms, device=None, sampling: bool = True):
        return check_batch(self.k, self.vocab, self.torch_dtype, self.max_batch, device or self.device, target, draft,
                           tokens, temperature, uniforms, need_tokens=sampling, need_uniforms=sampling)

    def _check_outputs(self, out, B, device=None, required=("tokens", "tau")):
        check_outputs(out, B, self.k, self.vocab, self.torch_dtype, device or self.device, required)

    def verify(self, target, draft, tokens, temperature, uniforms, want_pq: bool = True, want_tv: bool = False,
               out: dict | None = None, stream=None, want_entropy: bool = False) -> dict:
        """Verify a batch of chains held in CUDA tensors; returns output tensors (asynchronous).
        With want_entropy (or entropy tensors in `out`) this is spec_verify_ex, which also
        writes the entropy of every target and draft row."""
        B = self._check_inputs(target, draft, tokens, temperature, uniforms)
        if out is None:
            out = self.alloc_outputs(B, want_pq, want_tv, device=target.device, want_entropy=want_entropy)
        self._check_outputs(out, B)
        if (out.get("entropy_target") is None) != (out.get("entropy_draft") is None):
            raise ValueError("entropy_target and entropy_draft go together")
        args = (self._h, B, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(temperature), _ptr(uniforms),
                _ptr(out["tokens"]), _ptr(out["tau"]), _ptr(out.get("p_draft")), _ptr(out.get("q_draft")),
                _ptr(out.get("tv")))
        if "entropy_target" in out or "entropy_draft" in out:
            rc = self._lib.spec_verify_ex(*args, _ptr(out.get("entropy_target")), _ptr(out.get("entropy_draft")),
                                          self._stream(stream))
            _check(rc, "spec_verify_ex")
        else:
            rc = self._lib.spec_verify(*args, self._stream(stream))
            _check(rc, "spec_verify")
        return out

    def verify_lazy(self, target, draft, tokens, temperature, uniforms, out: dict | None = None, stream=None) -> dict:
        """spec_verify_lazy: verification that reads no row past a chain's first
        rejection (tokens and tau only; no p, q or TV)."""
        B = self._check_inputs(target, draft, tokens, temperature, uniforms)
        if out is None:
            out = self.alloc_outputs(B, want_pq=False, want_tv=False, device=target.device)
        self._check_outputs(out, B)
        rc = self._lib.spec_verify_lazy(self._h, B, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(temperature),
                                        _ptr(uniforms), _ptr(out["tokens"]), _ptr(out["tau"]), self._stream(stream))
        _check(rc, "spec_verify_lazy")
        return out

    def loss_grad(self, target, draft, temperature, kind: str = "overlap", weights=None, out: dict | None = None,
                  stream=None) -> dict:
        """spec_verify_loss_grad: per-position loss (kind "tv": 1 - alpha, "overlap":
        -ln alpha, alpha = sum min(p, q)) [B, k] fp32 and the gradient of the weighted
        loss with respect to the draft logits [B, k, V] in the logit dtype."""
        import torch
        B = self._check_inputs(target, draft, None, temperature, None, sampling=False)
        if kind not in ("tv", "overlap"):
            raise ValueError(f"kind must be 'tv' or 'overlap', not {kind!r}")
        code = {"tv": SV_LOSS_TV, "overlap": SV_LOSS_OVERLAP}[kind]
        if weights is not None:
            _check_tensor(weights, "weights", torch.float32, (B, self.k), self.device)
        if out is None:
            out = {"loss": torch.empty((B, self.k), dtype=torch.float32, device=target.device),
                   "grad": torch.empty_like(draft)}
        self._check_outputs(out, B, required=("grad",))
        rc = self._lib.spec_verify_loss_grad(self._h, B, _ptr(target), _ptr(draft), _ptr(temperature), code,
                                             _ptr(weights), _ptr(out.get("loss")), _ptr(out["grad"]),
                                             self._stream(stream))
        _check(rc, "spec_verify_loss_grad")
        return out

    def verify_tv(self, target, draft, temperature, out=None, stream=None):
        """Per-position TV distance only ([B, k] fp32)."""
        import torch
        B = self._check_inputs(target, draft, None, temperature, None, sampling=False)
        if out is None:
            out = torch.empty((B, self.k), dtype=torch.float32, device=target.device)
        _check_tensor(out, "out", torch.float32, (B, self.k), self.device)
        rc = self._lib.spec_verify_tv(self._h, B, _ptr(target), _ptr(draft), _ptr(temperature), _ptr(out),
                                      self._stream(stream))
        _check(rc, "spec_verify_tv")
        return out

    def verify_host(self, target, draft, tokens, temperature, uniforms, out: dict, stream=None) -> dict:
        """spec_verify_host: host tensors in and out; the handle needs
        SV_FLAG_HOST_STAGING.  Pinned logits are read in place by the kernels,
        pageable ones copied to the device first.  Synchronise the stream
        before reading out."""
        import torch
        cpu = torch.device("cpu")
        B = self._check_inputs(target, draft, tokens, temperature, uniforms, device=cpu)
        self._check_outputs(out, B, device=cpu)
        rc = self._lib.spec_verify_host(self._h, B, _ptr(target), _ptr(draft), _ptr(tokens), _ptr(temperature),
                                        _ptr(uniforms), _ptr(out["tokens"]), _ptr(out["tau"]),
                                        _ptr(out.get("p_draft")), _ptr(out.get("q_draft")), _ptr(out.get("tv")),
                                        self._stream(stream))
        _check(rc, "spec_verify_host")
        return out

    def kernel_times(self, max_n: int = 4096) -> list:
        """Durations (ms) of the verification kernel of the calls since the last read
        (handle created with SV_FLAG_KERNEL_TIMING)."""
        buf = (ctypes.c_float * max_n)()
        n = ctypes.c_int(0)
        _check(self._lib.spec_verify_kernel_times(self._h, buf, max_n, ctypes.byref(n)), "spec_verify_kernel_times")
        return list(buf[:n.value])

    def selftest_wait(self, polls: int):
        """spec_verify_selftest_wait: (status, [cycles of the first wait, of the second])."""
        c = (ctypes.c_longlong * 2)()
        rc = self._lib.spec_verify_selftest_wait(self._h, int(polls), c)
        return rc, [c[0], c[1]]

    def get_error(self):
        """Synchronise; return (status, invalid_count) and clear the device flags."""
        n = ctypes.c_int(0)
        rc = self._lib.spec_verify_get_error(self._h, ctypes.byref(n))
        return rc, n.value


__all__ = ["SpecVerifier", "SpecVerifyError", "build", "check_batch", "check_outputs", "output_shapes", "SV_FP32", "SV_BF16", "SV_FLAG_HOST_STAGING",
           "SV_FLAG_NO_TMA", "SV_FLAG_KERNEL_TIMING", "SV_OK", "SV_ERR_DATA", "SV_ERR_ARG", "SV_ERR_TIMEOUT"]
