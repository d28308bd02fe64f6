"""spec_verify_noalloc, the entry point for callers that cannot allocate device
memory (cudaMalloc can synchronise the device, and an engine that reserved its
memory at start-up may refuse new allocations).  It keeps its workspace in a
static device array, so it needs no handle.  Its outputs must match those of
spec_verify (the handle-based entry point) on the same inputs, on two calls in
a row that share that array.

Kept in a file that pytest collects last, so a run that stops at the first
failure has already run every other test."""
import ctypes
import json
import os
import subprocess
import sys

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


# Run in a fresh process: the library's module is loaded (its static array and
# the kernels' code placed on the device) by a handle that runs one call and is
# closed again, so that the first allocation-free call, with its one-time
# set-up, is the only thing between the two readings of the device's free
# memory.
_FRESH = r"""
import ctypes, json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import spec_inputs as si
import speculative_decoding_verification_68_gb300 as sv
from speculative_decoding_verification_68_gb300 import _native
lib = _native.load()
w = si.C3_T1.scaled(batch=24)
b = si.generate(w)
dev = torch.device("cuda")
ins = (torch.from_numpy(b.target.view(np.int16)).to(dev).view(torch.bfloat16),
       torch.from_numpy(b.draft.view(np.int16)).to(dev).view(torch.bfloat16),
       torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev), torch.from_numpy(b.uniforms).to(dev))
h = sv.SpecVerifier(24, w.k, w.vocab, torch.bfloat16)
out = h.alloc_outputs(24, want_pq=True, want_tv=True)
h.verify(*ins, want_tv=True)   # the kernels' code is placed on the device at their first launch
h.verify_lazy(*ins)            # (and the driver's memset kernel)
torch.cuda.synchronize()
h.close()
stream = torch.cuda.current_stream()
p = lambda t: ctypes.c_void_p(t.data_ptr())
torch.cuda.synchronize()
free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
rc = lib.spec_verify_noalloc(24, w.k, w.vocab, sv.SV_BF16, *[p(t) for t in ins], p(out["tokens"]), p(out["tau"]),
                             p(out["p_draft"]), p(out["q_draft"]), p(out["tv"]), ctypes.c_void_p(stream.cuda_stream))
torch.cuda.synchronize()
free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
ref = sv.SpecVerifier(24, w.k, w.vocab, torch.bfloat16)
want = ref.verify(*ins, want_tv=True)
torch.cuda.synchronize()
same = all(np.array_equal(out[k].cpu().numpy(), want[k].cpu().numpy()) for k in ("tokens", "tau"))
print(json.dumps({"rc": rc, "free0": free0, "free1": free1, "alloc0": alloc0, "alloc1": alloc1, "same": same}))
"""


def test_noalloc_first_call_allocates_nothing():
    """In a fresh process, the device's free memory (and the caching
    allocator's count) is the same before and after the first allocation-free
    call, which includes its one-time set-up."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    sv.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["rc"] == 0 and res["same"], res
    assert res["free1"] == res["free0"], res
    assert res["alloc1"] == res["alloc0"], res
