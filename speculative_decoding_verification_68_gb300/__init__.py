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

    def _check_inputs(self, target, draft, tokens, temperature, uniforms):
        import torch
        B = target.shape[0]
        k, V = self.k, self.vocab
        assert target.dtype == self.torch_dtype and draft.dtype == self.torch_dtype, "logit dtype mismatch"
        assert tuple(target.shape) == (B, k + 1, V) and tuple(draft.shape) == (B, k, V), "logit shape mismatch"
        assert target.is_contiguous() and draft.is_contiguous()
        if tokens is not None:
            assert tokens.dtype == torch.int32 and tuple(tokens.shape) == (B, k) and tokens.is_contiguous()
        assert temperature.dtype == torch.float32 and tuple(temperature.shape) == (B,)
        if uniforms is not None:
            assert uniforms.dtype == torch.float32 and tuple(uniforms.shape) == (B, k + 1) and uniforms.is_contiguous()
        return B

    def verify(self, target, draft, tokens, temperature, uniforms, want_pq: bool = True, want_tv: bool = False,
               out: dict | None = None, stream=None, want_entropy: bool = False) -> dict:
        """Verify a batch of chains held in CUDA tensors; returns output tensors (asynchronous).
        With want_entropy (or entropy tensors in `out`) this is spec_verify_ex, which also
        writes the entropy of every target and draft row."""
        B = self._check_inputs(target, draft, tokens, temperature, uniforms)
        if out is None:
            out = self.alloc_outputs(B, want_pq, want_tv, device=target.device, want_entropy=want_entropy)
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
        B = self._check_inputs(target, draft, None, temperature, None)
        code = {"tv": SV_LOSS_TV, "overlap": SV_LOSS_OVERLAP}[kind]
        if weights is not None:
            assert weights.dtype == torch.float32 and tuple(weights.shape) == (B, self.k) and weights.is_contiguous()
        if out is None:
            out = {"loss": torch.empty((B, self.k), dtype=torch.float32, device=target.device),
                   "grad": torch.empty_like(draft)}
        rc = self._lib.spec_verify_loss_grad(self._h, B, _ptr(target), _ptr(draft), _ptr(temperature), code,
                                             _ptr(weights), _ptr(out.get("loss")), _ptr(out["grad"]),
                                             self._stream(stream))
        _check(rc, "spec_verify_loss_grad")
        return out

    def verify_tv(self, target, draft, temperature, out=None, stream=None):
        """Per-position TV distance only ([B, k] fp32)."""
        import torch
        B = self._check_inputs(target, draft, None, temperature, None)
        if out is None:
            out = torch.empty((B, self.k), dtype=torch.float32, device=target.device)
        rc = self._lib.spec_verify_tv(self._h, B, _ptr(target), _ptr(draft), _ptr(temperature), _ptr(out),
                                      self._stream(stream))
        _check(rc, "spec_verify_tv")
        return out

    def verify_host(self, target, draft, tokens, temperature, uniforms, out: dict, stream=None) -> dict:
        """spec_verify_host: host tensors in and out; the handle needs
        SV_FLAG_HOST_STAGING.  Pinned logits are read in place by the kernels,
        pageable ones copied to the device first.  Synchronise the stream
        before reading out."""
        B = self._check_inputs(target, draft, tokens, temperature, uniforms)
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


__all__ = ["SpecVerifier", "SpecVerifyError", "build", "SV_FP32", "SV_BF16", "SV_FLAG_HOST_STAGING",
           "SV_FLAG_NO_TMA", "SV_FLAG_KERNEL_TIMING", "SV_OK", "SV_ERR_DATA", "SV_ERR_ARG", "SV_ERR_TIMEOUT"]
