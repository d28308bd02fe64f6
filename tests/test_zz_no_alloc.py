"""spec_verify_noalloc, the entry point for callers that cannot allocate device
memory (cudaMalloc can synchronise the device, and an engine that reserved its
memory at start-up may refuse new allocations).  It keeps its workspace in a
static device array, so it needs no handle.  Its outputs must match those of
spec_verify (the handle-based entry point) on the same inputs, on two calls in
a row that share that array.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import spec_inputs as si
from tests import _parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _dev(b):
    dev = torch.device("cuda")
    if b.workload.dtype == si.BF16:
        tgt = torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16)
        dft = torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tgt = torch.from_numpy(b.target).to(dev)
        dft = torch.from_numpy(b.draft).to(dev)
    return (tgt, dft, torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev),
            torch.from_numpy(b.uniforms).to(dev))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_matches_spec_verify_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    from speculative_decoding_verification_68_gb300 import _native
    sv.build()
    lib = _native.load()
    w = si.C3_T1.scaled(batch=24)
    # two different batches: the second call runs on whatever the first left in the array
    batches = [si.generate(w.scaled(seed=1)), si.generate(w.scaled(seed=2))]
    ref = sv.SpecVerifier(24, w.k, w.vocab, torch.bfloat16)
    stream = torch.cuda.current_stream()
    for b in batches:
        inputs = _dev(b)
        want = ref.verify(*inputs, want_tv=True)
        got = ref.alloc_outputs(24, want_pq=True, want_tv=True)
        rc = lib.spec_verify_noalloc(24, w.k, w.vocab, sv.SV_BF16, *[_ptr(t) for t in inputs],
                                     _ptr(got["tokens"]), _ptr(got["tau"]), _ptr(got["p_draft"]),
                                     _ptr(got["q_draft"]), _ptr(got["tv"]), ctypes.c_void_p(stream.cuda_stream))
        assert rc == sv.SV_OK, lib.spec_verify_strerror(rc)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in got.items()}
        r = {k: v.cpu().numpy() for k, v in want.items()}
        assert np.array_equal(g["tokens"], r["tokens"]) and np.array_equal(g["tau"], r["tau"])
        for key in ("p_draft", "q_draft"):
            assert np.all(np.abs(g[key] - r[key]) <= _parity.P_RTOL * np.abs(r[key]) + _parity.P_ATOL), key
        assert np.all(np.abs(g["tv"] - r["tv"]) <= _parity.TV_RTOL * r["tv"] + _parity.TV_ATOL)
    ref.close()
    # a batch beyond the static array is refused before any launch
    big = lib.spec_verify_noalloc(4000, w.k, w.vocab, sv.SV_BF16, *([None] * 10), ctypes.c_void_p(0))
    assert big == sv.SV_ERR_SIZE
