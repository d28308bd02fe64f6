"""Failure detection on the GPU without a fault: the kernels' bounded waits
give up on a barrier that nothing completes, flag the handle, and leave the
context usable (through the C ABI)."""
import numpy as np
import pytest

import spec_inputs as si
from tests import _parity

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_68_gb300 as sv
    sv.build()
    return sv


def test_bounded_waits_expire_and_context_survives(lib, oracle):
    w = si.C2
    v = lib.SpecVerifier(w.batch, w.k, w.vocab, torch.float32)
    polls = 1 << 12
    rc, cycles = v.selftest_wait(polls)
    assert rc == lib.SV_ERR_TIMEOUT, rc
    # the first wait polled to its limit; the second saw the flag and left within 256 polls
    assert cycles[0] > 0 and cycles[1] * 4 < cycles[0], cycles
    print(f"{cycles[0] / polls:.0f} cycles per poll: the kernels' 2^18-poll limit is about "
          f"{cycles[0] / polls * (1 << 18) / 2.07e9:.2f} s at 2.07 GHz")
    b = si.generate(w)
    dev = torch.device("cuda")
    ins = (torch.from_numpy(b.target).to(dev), torch.from_numpy(b.draft).to(dev),
           torch.from_numpy(b.tokens).to(dev), torch.from_numpy(b.temperature).to(dev),
           torch.from_numpy(b.uniforms).to(dev))
    # while the timeout flag is set, a call reports every chain invalid instead of
    # outputs computed after a wait gave up (no real wait expires here: the data arrives)
    out = v.verify(*ins, want_tv=True)
    torch.cuda.synchronize()
    assert np.all(out["tau"].cpu().numpy() == -1) and np.all(out["tokens"].cpu().numpy() == -1)
    assert np.all(np.isnan(out["tv"].cpu().numpy()))
    lz = v.verify_lazy(*ins)
    torch.cuda.synchronize()
    assert np.all(lz["tau"].cpu().numpy() == -1)
    assert v.get_error()[0] == lib.SV_ERR_TIMEOUT      # reported, and cleared
    assert v.get_error() == (lib.SV_OK, 0)
    # the same handle verifies correctly afterwards
    out = v.verify(*ins, want_tv=True)
    torch.cuda.synchronize()
    assert v.get_error() == (lib.SV_OK, 0)
    got = {k: t.cpu().numpy() for k, t in out.items()}
    ref = oracle.verify(b.target, b.draft, b.tokens, b.temperature, b.uniforms, w.dtype, nthreads=16)
    _parity.assert_parity(got, ref, w.k)
    v.close()
